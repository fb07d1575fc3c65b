// moe_permute.cu -- expert -> slot map, local-range mask/remap, per-slot
// histogram, exclusive scan and the stable token scatter.
//
// Method:
//  * Slot map -- TensorRT-LLM PR #4495 ("large-scale EP (part 3): refactor
//    FusedMoe for redundant expert"), Description: the fused op computes on
//    expert slots, into which the module loads the weights; expert id == slot id
//    until a mapping is introduced.  Replica table: expert e owns
//    rep_offset[e+1] - rep_offset[e] slots and token t uses replica t mod count.
//  * Local range -- vLLM EP FusedMoE patch, ep_mask_and_remap: local iff
//    start <= id < start + E_local; weights *= mask; local ids -> id - start;
//    non-local ids -> id mod E_local (MOD) or dropped (SKIP, the token-level
//    skip named in the same function's comments).
//  * Grouping -- the per-expert loop of the same patch's docstring (skip count
//    0): rows of a slot are contiguous, offsets are the exclusive scan of the
//    counts, and within a slot pairs keep ascending pair index t*k + j.
//
// Pipeline (no atomics decide any output position; results are deterministic):
//  K1 permute_count_kernel  one warp per chunk of 512 pairs: slot map + mask,
//                           writes slot_ids (and zeroes masked weights), and
//                           the chunk's per-slot counts.
//  K2 permute_scan_kernel   one CTA: counts = column sums, offsets = exclusive
//                           scan, base[c][s] = offsets[s] + sum of earlier
//                           chunks' counts of s.
//  K3 permute_place_kernel  one warp per chunk: walks its pairs in order, 32 at
//                           a time; lanes with equal slots are ranked with
//                           __match_any_sync, so row = base + running count +
//                           rank among lower lanes.  Writes pair_row, perm_src.
//  K4 permute_gather_kernel one warp per row: x_perm[r] = x[perm_src[r] / k]
//                           with 16-byte loads/stores.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int PM_CHUNK = 512;     // pairs per warp-chunk
constexpr int PM_WARPS = 8;       // warps per CTA in K1 / K3
constexpr int PM_SCAN_THREADS = 1024;

__device__ __forceinline__ int32_t map_slot(int32_t e, int64_t t, int E, const int32_t* __restrict__ rep_offset,
                                            const int32_t* __restrict__ rep_slots, int S, int32_t* status) {
    if (e < 0 || e >= E) {
        report(status, MOE_ERR_DEVICE_BOUNDS);
        return -1;
    }
    if (!rep_offset) return e;
    const int32_t lo = rep_offset[e];
    const int32_t cnt = rep_offset[e + 1] - lo;
    if (cnt <= 0 || lo < 0 || lo + cnt > S) {
        report(status, MOE_ERR_DEVICE_BOUNDS);
        return -1;
    }
    const int32_t s = rep_slots[lo + (int32_t)(t % cnt)];
    if (s < 0 || s >= S) {
        report(status, MOE_ERR_DEVICE_BOUNDS);
        return -1;
    }
    return s;
}

__global__ void __launch_bounds__(PM_WARPS * 32) permute_count_kernel(
    const int32_t* __restrict__ ids, float* __restrict__ w, int64_t P, int k, int E,
    const int32_t* __restrict__ rep_offset, const int32_t* __restrict__ rep_slots, int S, int local_start,
    int local_count, int mode, int S_local, int32_t* __restrict__ slot_ids, int32_t* __restrict__ chunk_cnt,
    int64_t nchunks, int32_t* status) {
    extern __shared__ int32_t pm_cnt[];  // [PM_WARPS][S_local]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* cnt = pm_cnt + (size_t)warp * S_local;
    for (int s = lane; s < S_local; s += 32) cnt[s] = 0;
    __syncwarp();
    const int64_t c = (int64_t)blockIdx.x * PM_WARPS + warp;
    if (c >= nchunks) return;
    const int64_t p0 = c * PM_CHUNK;
    const int64_t p1 = min(P, p0 + PM_CHUNK);
    for (int64_t p = p0 + lane; p < p1; p += 32) {
        const int64_t t = p / k;
        int32_t s = map_slot(ids[p], t, E, rep_offset, rep_slots, S, status);
        if (s >= 0 && local_count >= 0) {
            const bool local = (s >= local_start) && (s < local_start + local_count);
            w[p] = w[p] * (local ? 1.0f : 0.0f);
            s = local ? s - local_start : (mode == MOE_NONLOCAL_MOD ? s % local_count : -1);
        } else if (s < 0 && local_count >= 0) {
            w[p] = w[p] * 0.0f;
        }
        slot_ids[p] = s;
        if (s >= 0) atomicAdd(&cnt[s], 1);
    }
    __syncwarp();
    int32_t* dst = chunk_cnt + c * S_local;
    for (int s = lane; s < S_local; s += 32) dst[s] = cnt[s];
}

__global__ void __launch_bounds__(PM_SCAN_THREADS) permute_scan_kernel(const int32_t* __restrict__ chunk_cnt,
                                                                       int64_t nchunks, int S_local,
                                                                       int32_t* __restrict__ counts,
                                                                       int32_t* __restrict__ offsets,
                                                                       int32_t* __restrict__ chunk_base) {
    __shared__ int32_t s_warp[PM_SCAN_THREADS / 32];
    const int s = threadIdx.x;
    int32_t tot = 0;
    if (s < S_local) {
        for (int64_t c = 0; c < nchunks; ++c) tot += chunk_cnt[c * S_local + s];
        counts[s] = tot;
    }
    // block exclusive scan of tot over s
    const int lane = s & 31, warp = s >> 5;
    int32_t incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t v = (lane < PM_SCAN_THREADS / 32) ? s_warp[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        s_warp[lane] = v;  // inclusive prefix over warps
    }
    __syncthreads();
    const int32_t excl = incl - tot + (warp > 0 ? s_warp[warp - 1] : 0);
    if (s < S_local) {
        offsets[s] = excl;
        int32_t run = excl;
        for (int64_t c = 0; c < nchunks; ++c) {
            chunk_base[c * S_local + s] = run;
            run += chunk_cnt[c * S_local + s];
        }
        if (s == S_local - 1) offsets[S_local] = excl + tot;
    }
}

__global__ void __launch_bounds__(PM_WARPS * 32) permute_place_kernel(const int32_t* __restrict__ slot_ids,
                                                                      int64_t P, int S_local,
                                                                      const int32_t* __restrict__ chunk_base,
                                                                      int64_t nchunks,
                                                                      int32_t* __restrict__ pair_row,
                                                                      int32_t* __restrict__ perm_src) {
    extern __shared__ int32_t pm_cur[];  // [PM_WARPS][S_local]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * PM_WARPS + warp;
    if (c >= nchunks) return;
    int32_t* cur = pm_cur + (size_t)warp * S_local;
    for (int s = lane; s < S_local; s += 32) cur[s] = chunk_base[c * S_local + s];
    __syncwarp();
    const int64_t p0 = c * PM_CHUNK;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int it = 0; it < PM_CHUNK / 32; ++it) {
        const int64_t p = p0 + it * 32 + lane;
        if (p0 + it * 32 >= P) break;
        const int32_t s = (p < P) ? slot_ids[p] : -2;
        const uint32_t peers = __match_any_sync(0xffffffffu, s);
        if (s >= 0) {
            const int32_t row = cur[s] + __popc(peers & lt_mask);
            pair_row[p] = row;
            perm_src[row] = (int32_t)p;
        } else if (s == -1) {
            pair_row[p] = -1;
        }
        __syncwarp();
        if (s >= 0 && lane == 31 - __clz(peers)) cur[s] += __popc(peers);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(256) permute_gather_kernel(const uint16_t* __restrict__ x,
                                                             const int32_t* __restrict__ perm_src,
                                                             const int32_t* __restrict__ offsets, int S_local,
                                                             int k, int H, int64_t P, uint16_t* __restrict__ x_perm,
                                                             int32_t* status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t rows = offsets[S_local];
    const int vec = H / 8;
    for (int64_t r = (int64_t)blockIdx.x * 8 + warp; r < rows; r += (int64_t)gridDim.x * 8) {
        const int32_t p = perm_src[r];
        if (p < 0 || p >= P) {
            if (lane == 0) report(status, MOE_ERR_DEVICE_BOUNDS);
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)(p / k) * H);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + r * H);
        for (int v = lane; v < vec; v += 32) dst[v] = __ldg(src + v);
    }
}

}  // namespace

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t permute_scratch_bytes(int64_t P, int S_local) {
    const int64_t nchunks = (P + PM_CHUNK - 1) / PM_CHUNK;
    return 2 * align256((size_t)std::max<int64_t>(nchunks, 1) * (size_t)S_local * sizeof(int32_t));
}

void permute_carve(void* base, int64_t P, int S_local, int32_t** chunk_cnt, int32_t** chunk_base) {
    const int64_t nchunks = (P + PM_CHUNK - 1) / PM_CHUNK;
    const size_t one = align256((size_t)std::max<int64_t>(nchunks, 1) * (size_t)S_local * sizeof(int32_t));
    *chunk_cnt = static_cast<int32_t*>(base);
    *chunk_base = reinterpret_cast<int32_t*>(static_cast<char*>(base) + one);
}

cudaError_t launch_permute(const PermuteLaunch& L, int num_sms, cudaStream_t s) {
    const int64_t P = L.T * L.k;
    const int64_t nchunks = (P + PM_CHUNK - 1) / PM_CHUNK;
    const unsigned g13 = (unsigned)((nchunks + PM_WARPS - 1) / PM_WARPS);
    const size_t smem = (size_t)PM_WARPS * L.S_local * sizeof(int32_t);
    int32_t* status = &L.hdr->status;
    permute_count_kernel<<<g13, PM_WARPS * 32, smem, s>>>(L.ids, L.w, P, L.k, L.E, L.rep_offset, L.rep_slots, L.S,
                                                          L.local_start, L.local_count, L.mode, L.S_local,
                                                          L.slot_ids, L.chunk_cnt, nchunks, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    permute_scan_kernel<<<1, PM_SCAN_THREADS, 0, s>>>(L.chunk_cnt, nchunks, L.S_local, L.counts, L.offsets,
                                                      L.chunk_base);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    permute_place_kernel<<<g13, PM_WARPS * 32, smem, s>>>(L.slot_ids, P, L.S_local, L.chunk_base, nchunks,
                                                          L.pair_row, L.perm_src);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int64_t want = (P + 7) / 8;
    const unsigned g4 = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    permute_gather_kernel<<<g4, 256, 0, s>>>(L.x, L.perm_src, L.offsets, L.S_local, L.k, L.H, P, L.x_perm, status);
    return cudaGetLastError();
}

}  // namespace moe
