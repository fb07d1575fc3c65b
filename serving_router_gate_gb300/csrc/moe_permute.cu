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
//  1 rank    one warp per chunk of 256 pairs: slot map + mask (writes
//            slot_ids, zeroes masked weights), then the stable rank of each
//            pair among the chunk's pairs of its slot (__match_any_sync over 32
//            lanes plus a per-warp running count), and the chunk's counts.
//  2 scan    one CTA: counts = column sums, offsets = exclusive scan,
//            base[c][s] = offsets[s] + earlier chunks' counts of s.
//  3 scatter 8 pairs per warp step: row = base[chunk][slot] + rank; writes
//            pair_row and perm_src, and the warp copies x[t] into x_perm[row]
//            with 16-byte loads/stores (skipped when the caller passes no
//            x_perm: a consumer that reads the token rows through pair_row).
// Large batches run the phases as three kernels over the whole GPU; batches of
// at most 8192 pairs run phases 1-2 in one CTA (one launch) separated by
// barriers, and phase 3 too when its row copy is at most 256 KB.
#include <stdint.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int PM_CHUNK = 256;     // pairs per warp-chunk
constexpr int PM_ROUNDS = PM_CHUNK / 32;
constexpr int PM_WARPS = 8;       // warps per CTA in K1 / K3
constexpr int PM_SCAN_THREADS = 1024;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

// ---- the three phases, as device functions shared by the multi-CTA kernels
// and the one-CTA kernel for small batches ----

// Phase 1, one warp on chunk c (pairs c*PM_CHUNK ..): slot map + mask (writes
// slot_ids, zeroes masked weights), the stable rank of each pair among the
// chunk's pairs of its slot, and the chunk's per-slot counts.  `cur` is this
// warp's S_local shared-memory counters.
__device__ __forceinline__ void rank_chunk(int64_t c, const int32_t* __restrict__ ids, float* __restrict__ w,
                                           int64_t P, int k, int E, const int32_t* __restrict__ rep_offset,
                                           const int32_t* __restrict__ rep_slots, int S, int local_start,
                                           int local_count, int mode, int S_local, int32_t* __restrict__ slot_ids,
                                           int32_t* __restrict__ rank, int32_t* __restrict__ chunk_cnt,
                                           int32_t* cur, int32_t* status) {
    const int lane = threadIdx.x & 31;
    for (int s = lane; s < S_local; s += 32) cur[s] = 0;
    __syncwarp();
    const int64_t p0 = c * PM_CHUNK;
    int32_t sl[PM_ROUNDS];
#pragma unroll
    for (int r = 0; r < PM_ROUNDS; ++r) {  // all loads in flight before any use
        const int64_t p = p0 + r * 32 + lane;
        sl[r] = (p < P) ? ids[p] : INT32_MIN;
    }
#pragma unroll
    for (int r = 0; r < PM_ROUNDS; ++r) {
        const int64_t p = p0 + r * 32 + lane;
        if (p >= P) {
            sl[r] = -2;  // padding lane: neither counted nor written
            continue;
        }
        int32_t s = map_slot(sl[r], p / k, E, rep_offset, rep_slots, S, status);
        if (local_count >= 0) {
            const bool local = (s >= local_start) && (s < local_start + local_count);
            w[p] = w[p] * (local ? 1.0f : 0.0f);
            if (s >= 0) s = local ? s - local_start : (mode == MOE_NONLOCAL_MOD ? s % local_count : -1);
        }
        slot_ids[p] = s;
        sl[r] = s;
    }
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < PM_ROUNDS; ++r) {
        const int32_t s = sl[r];
        const uint32_t peers = __match_any_sync(0xffffffffu, s);
        if (s >= 0) rank[p0 + r * 32 + lane] = cur[s] + __popc(peers & lt_mask);
        __syncwarp();
        if (s >= 0 && lane == 31 - __clz(peers)) cur[s] += __popc(peers);
        __syncwarp();
    }
    int32_t* dst = chunk_cnt + c * S_local;
    for (int s = lane; s < S_local; s += 32) dst[s] = cur[s];
}

// Phase 2, one CTA of PM_SCAN_THREADS threads: counts = column sums,
// offsets = exclusive scan, base[c][s] = offsets[s] + earlier chunks' counts.
__device__ __forceinline__ void scan_counts(const int32_t* __restrict__ chunk_cnt, int64_t nchunks, int S_local,
                                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ chunk_base, int32_t* s_warp) {
    const int s = threadIdx.x;
    int32_t tot = 0;
    if (s < S_local) {
        int64_t c = 0;
        for (; c + 4 <= nchunks; c += 4) {
            const int32_t a0 = chunk_cnt[(c + 0) * S_local + s], a1 = chunk_cnt[(c + 1) * S_local + s];
            const int32_t a2 = chunk_cnt[(c + 2) * S_local + s], a3 = chunk_cnt[(c + 3) * S_local + s];
            tot += a0 + a1 + a2 + a3;
        }
        for (; c < nchunks; ++c) tot += chunk_cnt[c * S_local + s];
        counts[s] = tot;
    }
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
            const int32_t v = chunk_cnt[c * S_local + s];
            chunk_base[c * S_local + s] = run;
            run += v;
        }
        if (s == S_local - 1) offsets[S_local] = excl + tot;
    }
}

// Phase 3, one warp on 8 pairs at pb: row = base[chunk][slot] + rank; lanes
// 0..7 write pair_row / perm_src, then the warp copies the 8 rows of x.
constexpr int PS_PAIRS = 8;

// bf16 of the exact product w * x (x a bf16 value), rounded once to nearest,
// ties to even: fp32 rounds the product to p with an exact remainder e = w*x - p
// (fma); bf16 rounding points are fp32 values, so p rounds like the exact
// product unless p sits exactly on a midpoint between two bf16 values, where
// the sign of e decides.
__device__ __forceinline__ uint32_t bf16_of_product(float w, float x) {
    const float p = __fmul_rn(w, x);
    const float e = fmaf(w, x, -p);
    const uint32_t b = __float_as_uint(p);
    if ((b & 0xFFFFu) == 0x8000u && e != 0.0f) {
        const uint32_t t = b & 0xFFFF0000u;  // toward zero
        return ((e > 0.0f) == (p > 0.0f) ? t + 0x10000u : t) >> 16;
    }
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(p));
}

// Copy (or, with wsc, scale by the pair's routing weight) the rows of pairs
// pb .. pb+7 into their x_perm rows (none when x_perm is null); also writes
// pair_row and perm_src.
__device__ __forceinline__ void scatter_pairs(int64_t pb, const uint16_t* __restrict__ x,
                                              const int32_t* __restrict__ slot_ids, const int32_t* __restrict__ rank,
                                              const int32_t* __restrict__ chunk_base, int S_local, int64_t P, int k,
                                              int H, int32_t* __restrict__ pair_row, int32_t* __restrict__ perm_src,
                                              uint16_t* __restrict__ x_perm, const float* __restrict__ wsc,
                                              int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int vec = H / 8;
    int32_t row = -1;
    float wp = 1.0f;
    if (lane < PS_PAIRS && pb + lane < P) {
        const int64_t p = pb + lane;
        const int32_t s = slot_ids[p];
        if (s >= 0) {
            row = chunk_base[(p / PM_CHUNK) * S_local + s] + rank[p];
            if (!in_bounds(row, P, status)) row = -1;
        }
        if (row >= 0) {
            perm_src[row] = (int32_t)p;
            if (wsc) wp = wsc[p];
        }
        pair_row[p] = row;
    }
    if (!x_perm) return;  // routing tables only
    const int nj = (int)min((int64_t)PS_PAIRS, P - pb);
    if (!wsc) {
        // the pairs of one token share its row: each 16-byte vector of the row is loaded
        // once (eight per lane in flight) and stored to every one of its pairs' rows
        int j0 = 0;
        while (j0 < nj) {
            const int64_t tok = (pb + j0) / k;
            int j1 = j0 + 1;
            while (j1 < nj && (pb + j1) / k == tok) ++j1;
            const uint4* src = reinterpret_cast<const uint4*>(x + tok * H);
            for (int v0 = lane; v0 < vec; v0 += 32 * 8) {
                uint4 buf[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + 32 * u;
                    if (v < vec) buf[u] = __ldg(src + v);
                }
                for (int j = j0; j < j1; ++j) {
                    const int32_t r = __shfl_sync(0xffffffffu, row, j);
                    if (r < 0) continue;
                    uint4* dst = reinterpret_cast<uint4*>(x_perm + (int64_t)r * H);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int v = v0 + 32 * u;
                        if (v < vec) dst[v] = buf[u];
                    }
                }
            }
            j0 = j1;
        }
        return;
    }
    for (int j = 0; j < nj; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, row, j);
        const float wj = __shfl_sync(0xffffffffu, wp, j);
        if (r < 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(x + ((pb + j) / k) * H);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (int64_t)r * H);
        // routing on the input: each pair's row scaled by its own weight; unrolled so the
        // loads of several vectors are in flight before the first one's products are rounded
#pragma unroll 4
        for (int v = lane; v < vec; v += 32) {
            float f[8];
            unpack8(__ldg(src + v), f);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = bf16_of_product(wj, f[2 * i]) | (bf16_of_product(wj, f[2 * i + 1]) << 16);
            dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// ---- multi-CTA kernels ----

__global__ void __launch_bounds__(PM_WARPS * 32) permute_rank_kernel(
    const int32_t* __restrict__ ids, float* __restrict__ w, int64_t P, int k, int E,
    const int32_t* __restrict__ rep_offset, const int32_t* __restrict__ rep_slots, int S, int local_start,
    int local_count, int mode, int S_local, int32_t* __restrict__ slot_ids, int32_t* __restrict__ rank,
    int32_t* __restrict__ chunk_cnt, int64_t nchunks, int32_t* status) {
    extern __shared__ int32_t pm_cur[];  // [PM_WARPS][S_local]
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5;
    const int64_t c = (int64_t)blockIdx.x * PM_WARPS + warp;
    if (c >= nchunks) return;
    rank_chunk(c, ids, w, P, k, E, rep_offset, rep_slots, S, local_start, local_count, mode, S_local, slot_ids, rank,
               chunk_cnt, pm_cur + (size_t)warp * S_local, status);
}

__global__ void __launch_bounds__(PM_SCAN_THREADS) permute_scan_kernel(const int32_t* __restrict__ chunk_cnt,
                                                                       int64_t nchunks, int S_local,
                                                                       int32_t* __restrict__ counts,
                                                                       int32_t* __restrict__ offsets,
                                                                       int32_t* __restrict__ chunk_base) {
    __shared__ int32_t s_warp[PM_SCAN_THREADS / 32];
    pdl_wait();
    pdl_trigger();
    scan_counts(chunk_cnt, nchunks, S_local, counts, offsets, chunk_base, s_warp);
}

__global__ void __launch_bounds__(256) permute_scatter_kernel(const uint16_t* __restrict__ x,
                                                              const int32_t* __restrict__ slot_ids,
                                                              const int32_t* __restrict__ rank,
                                                              const int32_t* __restrict__ chunk_base, int S_local,
                                                              int64_t P, int k, int H,
                                                              int32_t* __restrict__ pair_row,
                                                              int32_t* __restrict__ perm_src,
                                                              uint16_t* __restrict__ x_perm,
                                                              const float* __restrict__ wsc, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5;
    for (int64_t pb = ((int64_t)blockIdx.x * 8 + warp) * PS_PAIRS; pb < P; pb += (int64_t)gridDim.x * 8 * PS_PAIRS)
        scatter_pairs(pb, x, slot_ids, rank, chunk_base, S_local, P, k, H, pair_row, perm_src, x_perm, wsc, status);
}

// ---- one CTA for small batches: the three phases with block barriers ----
constexpr int PM_SMALL_WARPS = PM_SCAN_THREADS / 32;  // 32 warps, one chunk each
constexpr int64_t PM_SMALL_MAX_P = (int64_t)PM_SMALL_WARPS * PM_CHUNK;
constexpr int PM_SMALL_MAX_S = 384;
constexpr int64_t PM_SMALL_COPY = 256 * 1024;  // row bytes one CTA copies itself

__global__ void __launch_bounds__(PM_SCAN_THREADS) permute_small_kernel(
    const int32_t* __restrict__ ids, float* __restrict__ w, int64_t P, int k, int E,
    const int32_t* __restrict__ rep_offset, const int32_t* __restrict__ rep_slots, int S, int local_start,
    int local_count, int mode, int S_local, int32_t* __restrict__ slot_ids, int32_t* __restrict__ rank,
    int32_t* __restrict__ chunk_cnt, int64_t nchunks, const uint16_t* __restrict__ x, int H,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ pair_row, int32_t* __restrict__ perm_src, uint16_t* __restrict__ x_perm,
    const float* __restrict__ wsc, int with_scatter, int32_t* status) {
    extern __shared__ int32_t pm_cur[];  // [32 warps][S_local]
    __shared__ int32_t s_warp[PM_SCAN_THREADS / 32];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5;
    if (warp < nchunks)
        rank_chunk(warp, ids, w, P, k, E, rep_offset, rep_slots, S, local_start, local_count, mode, S_local,
                   slot_ids, rank, chunk_cnt, pm_cur + (size_t)warp * S_local, status);
    __syncthreads();
    scan_counts(chunk_cnt, nchunks, S_local, counts, offsets, chunk_base, s_warp);
    if (!with_scatter) return;  // the rows are copied by permute_scatter_kernel over the whole GPU
    __syncthreads();
    for (int64_t pb = (int64_t)warp * PS_PAIRS; pb < P; pb += (int64_t)PM_SMALL_WARPS * PS_PAIRS)
        scatter_pairs(pb, x, slot_ids, rank, chunk_base, S_local, P, k, H, pair_row, perm_src, x_perm, wsc, status);
}

// ---- one CTA for tiny batches (at most one chunk of pairs): every phase in shared
// memory, no scratch in global memory ----
//
// The token rows are staged in shared memory while warp 0 maps, masks and ranks
// the pairs (as rank_chunk does, ranks kept in shared memory); the block then
// scans the counts, places every pair and writes the rows of x_perm from the
// staged copy.
constexpr int PT_THREADS = 512;
constexpr int PT_WARPS = PT_THREADS / 32;
constexpr int64_t PT_MAX_X_BYTES = 96 * 1024;

__global__ void __launch_bounds__(PT_THREADS) permute_tiny_kernel(
    const int32_t* __restrict__ ids, float* __restrict__ w, int T, int k, int E,
    const int32_t* __restrict__ rep_offset, const int32_t* __restrict__ rep_slots, int S, int local_start,
    int local_count, int mode, int S_local, const uint16_t* __restrict__ x, int H, int32_t* __restrict__ slot_ids,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ pair_row, uint16_t* __restrict__ x_perm, int scale_rows, int32_t* status) {
    extern __shared__ __align__(16) unsigned char pt_smem[];
    const size_t xb = x_perm ? (size_t)T * H * 2 : 0;                        // no rows staged without x_perm
    uint16_t* xs = reinterpret_cast<uint16_t*>(pt_smem);                      // [T][H]
    int32_t* cnt = reinterpret_cast<int32_t*>(pt_smem + xb);                  // [S_local]
    int32_t* off = cnt + S_local;                                             // [S_local]
    const int P = T * k;
    int32_t* s_slot = off + S_local;                                          // [P]
    int32_t* s_rank = s_slot + P;                                             // [P]
    int32_t* s_row = s_rank + P;                                              // [P]
    float* s_w = reinterpret_cast<float*>(s_row + P);                         // [P]
    __shared__ int32_t s_wsum[PT_WARPS];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    pdl_trigger();

    const int vec = H / 8;
    if (x_perm)
        for (int i = tid; i < T * vec; i += PT_THREADS) cp_async16(xs + (size_t)i * 8, x + (size_t)i * 8);
    cp_async_commit();
    for (int s = tid; s < S_local; s += PT_THREADS) cnt[s] = 0;
    __syncthreads();

    if (warp == 0) {
        // slot map + mask, then the stable rank of each pair among the pairs of its slot
        int32_t sl[PM_ROUNDS];
#pragma unroll
        for (int r = 0; r < PM_ROUNDS; ++r) {
            const int p = r * 32 + lane;
            sl[r] = p < P ? ids[p] : INT32_MIN;
        }
#pragma unroll
        for (int r = 0; r < PM_ROUNDS; ++r) {
            const int p = r * 32 + lane;
            if (p >= P) {
                sl[r] = -2;
                continue;
            }
            int32_t sv = map_slot(sl[r], p / k, E, rep_offset, rep_slots, S, status);
            float wp = w[p];
            if (local_count >= 0) {
                const bool local = (sv >= local_start) && (sv < local_start + local_count);
                wp = wp * (local ? 1.0f : 0.0f);
                w[p] = wp;
                if (sv >= 0) sv = local ? sv - local_start : (mode == MOE_NONLOCAL_MOD ? sv % local_count : -1);
            }
            slot_ids[p] = sv;
            s_slot[p] = sv;
            s_w[p] = wp;
            sl[r] = sv;
        }
        const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
        for (int r = 0; r < PM_ROUNDS; ++r) {
            const int32_t sv = sl[r];
            const uint32_t peers = __match_any_sync(0xffffffffu, sv);
            if (sv >= 0) s_rank[r * 32 + lane] = cnt[sv] + __popc(peers & lt_mask);
            __syncwarp();
            if (sv >= 0 && lane == 31 - __clz(peers)) cnt[sv] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();

    // counts and their exclusive scan: thread i takes slots 2i and 2i + 1
    const int s0 = 2 * tid;
    const int32_t c0 = s0 < S_local ? cnt[s0] : 0, c1 = s0 + 1 < S_local ? cnt[s0 + 1] : 0;
    int32_t incl = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int32_t before = 0;
    for (int i = 0; i < warp; ++i) before += s_wsum[i];
    const int32_t ex = before + incl - (c0 + c1);
    if (s0 < S_local) {
        counts[s0] = c0;
        offsets[s0] = ex;
        off[s0] = ex;
    }
    if (s0 + 1 < S_local) {
        counts[s0 + 1] = c1;
        offsets[s0 + 1] = ex + c0;
        off[s0 + 1] = ex + c0;
    }
    if (tid == PT_THREADS - 1) {
        int32_t total = 0;
        for (int i = 0; i < PT_WARPS; ++i) total += s_wsum[i];
        offsets[S_local] = total;
    }
    __syncthreads();

    for (int p = tid; p < P; p += PT_THREADS) {
        const int32_t sv = s_slot[p];
        int32_t row = sv >= 0 ? off[sv] + s_rank[p] : -1;
        if (row >= 0 && !in_bounds(row, P, status)) row = -1;
        pair_row[p] = row;
        if (row >= 0) perm_src[row] = p;
        s_row[p] = row;
    }
    cp_async_wait_group<0>();
    __syncthreads();

    // rows of x_perm from the staged token rows (or, with the routing applied on
    // the input, bf16(w * x))
    if (!x_perm) return;
    for (int f = tid; f < P * vec; f += PT_THREADS) {
        const int p = f / vec, v = f - p * vec;
        const int32_t row = s_row[p];
        if (row < 0) continue;
        const uint4 src = *reinterpret_cast<const uint4*>(xs + (size_t)(p / k) * H + (size_t)v * 8);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (int64_t)row * H) + v;
        if (!scale_rows) {
            *dst = src;
        } else {
            const float wj = s_w[p];
            float fx[8];
            unpack8(src, fx);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = bf16_of_product(wj, fx[2 * i]) | (bf16_of_product(wj, fx[2 * i + 1]) << 16);
            *dst = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t permute_scratch_bytes(int64_t P, int S_local) {
    const int64_t nchunks = (P + PM_CHUNK - 1) / PM_CHUNK;
    return align256((size_t)std::max<int64_t>(P, 1) * sizeof(int32_t)) +
           2 * align256((size_t)std::max<int64_t>(nchunks, 1) * (size_t)S_local * sizeof(int32_t));
}

void permute_carve(void* base, int64_t P, int S_local, int32_t** rank, int32_t** chunk_cnt, int32_t** chunk_base) {
    const int64_t nchunks = (P + PM_CHUNK - 1) / PM_CHUNK;
    const size_t r = align256((size_t)std::max<int64_t>(P, 1) * sizeof(int32_t));
    const size_t one = align256((size_t)std::max<int64_t>(nchunks, 1) * (size_t)S_local * sizeof(int32_t));
    char* b = static_cast<char*>(base);
    *rank = reinterpret_cast<int32_t*>(b);
    *chunk_cnt = reinterpret_cast<int32_t*>(b + r);
    *chunk_base = reinterpret_cast<int32_t*>(b + r + one);
}

cudaError_t launch_permute(const PermuteLaunch& L, int num_sms, cudaStream_t s) {
    // routing applied on the input: rows scaled by the (masked) weights
    const float* wsc = L.scale_rows ? L.w : nullptr;
    const int64_t P = L.T * L.k;
    const int64_t nchunks = (P + PM_CHUNK - 1) / PM_CHUNK;
    int32_t* status = &L.hdr->status;
    if (P <= PM_CHUNK && L.S_local <= 2 * PT_THREADS && L.T * (int64_t)L.H * 2 <= PT_MAX_X_BYTES) {
        const size_t smem = (L.x_perm ? (size_t)L.T * L.H * 2 : 0) + (size_t)2 * L.S_local * sizeof(int32_t) +
                            (size_t)4 * P * sizeof(int32_t);
        cudaError_t e = cudaFuncSetAttribute(permute_tiny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        return launch_k("permute_tiny", permute_tiny_kernel, dim3(1), dim3(PT_THREADS), smem, s, L.ids, L.w,
                        (int)L.T, L.k, L.E, L.rep_offset, L.rep_slots, L.S, L.local_start, L.local_count, L.mode,
                        L.S_local, L.x, L.H, L.slot_ids, L.counts, L.offsets, L.perm_src, L.pair_row, L.x_perm,
                        (int)L.scale_rows, status);
    }
    if (P <= PM_SMALL_MAX_P && L.S_local <= PM_SMALL_MAX_S) {
        const size_t smem_small = (size_t)PM_SMALL_WARPS * L.S_local * sizeof(int32_t);
        if (smem_small > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(permute_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem_small);
            if (e != cudaSuccess) return e;
        }
        // one CTA copies at most PM_SMALL_COPY bytes of rows; more go to the scatter kernel
        const bool copy_here = !L.x_perm || (int64_t)P * L.H * 2 <= PM_SMALL_COPY;
        cudaError_t e = launch_k("permute_small", permute_small_kernel, dim3(1), dim3(PM_SCAN_THREADS), smem_small,
                                 s, L.ids, L.w, P, L.k, L.E, L.rep_offset, L.rep_slots, L.S, L.local_start, L.local_count, L.mode,
                                 L.S_local, L.slot_ids, L.rank, L.chunk_cnt, nchunks, L.x, L.H, L.counts, L.offsets,
                                 L.chunk_base, L.pair_row, L.perm_src, L.x_perm, wsc, (int)copy_here, status);
        if (e != cudaSuccess || copy_here) return e;
        const int64_t want = (P + 8 * PS_PAIRS - 1) / (8 * PS_PAIRS);
        const unsigned gs = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
        return launch_k("permute_scatter", permute_scatter_kernel, dim3(gs), dim3(256), 0, s, L.x, L.slot_ids,
                        L.rank, L.chunk_base, L.S_local, P, L.k, L.H, L.pair_row, L.perm_src, L.x_perm, wsc, status);
    }
    const unsigned g1 = (unsigned)((nchunks + PM_WARPS - 1) / PM_WARPS);
    const size_t smem = (size_t)PM_WARPS * L.S_local * sizeof(int32_t);
    cudaError_t err = launch_k("permute_rank", permute_rank_kernel, dim3(g1), dim3(PM_WARPS * 32), smem, s, L.ids,
                               L.w, P, L.k, L.E, L.rep_offset, L.rep_slots, L.S, L.local_start, L.local_count, L.mode, L.S_local,
                               L.slot_ids, L.rank, L.chunk_cnt, nchunks, status);
    if (err != cudaSuccess) return err;
    err = launch_k("permute_scan", permute_scan_kernel, dim3(1), dim3(PM_SCAN_THREADS), 0, s, L.chunk_cnt, nchunks,
                   L.S_local, L.counts, L.offsets, L.chunk_base);
    if (err != cudaSuccess) return err;
    const int64_t want = (P + 8 * PS_PAIRS - 1) / (8 * PS_PAIRS);
    const unsigned g3 = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    return launch_k("permute_scatter", permute_scatter_kernel, dim3(g3), dim3(256), 0, s, L.x, L.slot_ids, L.rank,
                    L.chunk_base, L.S_local, P, L.k, L.H, L.pair_row, L.perm_src, L.x_perm, wsc, status);
}

}  // namespace moe
