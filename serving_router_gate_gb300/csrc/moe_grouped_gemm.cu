// moe_grouped_gemm.cu -- grouped GEMMs of the MoE experts on the tcgen05
// tensor cores (sm_103a): FC1 with a fused SwiGLU epilogue, and FC2.
//
// Method: per expert slot, the gated MLP (SwiGLU) of the TensorRT-LLM
// AutoDeploy MoE ops (PR #10985, "MoE all-to-all paradigm": is_gated_mlp and
// act_fn per expert); slots with no rows get no tiles (vLLM EP FusedMoE patch,
// module docstring: the per-expert loop skips experts with count 0).
//
// Design (one CTA per SM, persistent, 192 threads):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] (bf16,
//               128-byte swizzle) per K step into a 4-stage shared-memory ring.
//               FC1 loads the B tile as two 128-row halves -- gate rows n0.. and
//               up rows I+n0.. -- so one MMA of N = 256 yields matching gate
//               and up columns, with no weight re-layout.
//   warp 1      tensor memory allocator (512 columns = 2 accumulators of
//               256 fp32 columns) and, on one thread, the MMA issuer:
//               tcgen05.mma.cta_group::1.kind::f16 M=128 N=256 K=16, four per
//               K step, completion signalled through tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31 = tile rows), FC1: h = bf16(silu(gate) * up);
//               FC2: y = bf16(acc); 16-byte stores; rows past the slot's count
//               are not stored.  Two accumulators let the epilogue of one tile
//               overlap the main loop of the next.
// Tiles: an optional dense "shared expert" problem (M = T) first, then the
// routed problem, whose ragged per-slot row counts are read on the device from
// the offsets array (no host synchronisation): slot g has ceil(M_g / 128)
// m-tiles; within a slot, tiles run n-tile-major so consecutive CTAs share the
// same weight tile through L2.  Every wait is bounded: on a timeout the CTA
// records MOE_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees its
// tensor memory and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;            // MMA N
constexpr int BK = 64;             // bf16 elements per 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct GemmParams {
    const int32_t* offsets;  // [G+1] routed row offsets (device)
    int G;                   // routed groups (0: none)
    int K, K_sh;             // reduction lengths
    int N_out, N_out_sh;     // output columns
    int up_off, up_off_sh;   // FC1: first up row inside B
    int64_t rows_cap;        // rows of the routed A / output
    int64_t T_sh;            // rows of the shared problem (0: none)
    uint16_t* out;
    uint16_t* out_sh;
    int32_t* status;
    uint64_t timeout_ns;
};

struct SmemMeta {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int routed_tiles;
    int off[MAX_GROUPS + 1];
    int ts[MAX_GROUPS + 1];
};

constexpr size_t SMEM_BYTES = 1024 /*alignment slack*/ + (size_t)STAGES * STAGE_BYTES + sizeof(SmemMeta);

struct Tile {
    int prob;        // 0 routed, 1 shared
    int g;           // routed group
    int nt;          // n-tile
    int row0;        // first row in A / out
    int rows_valid;  // rows of this tile that belong to the group
};

template <bool kFC1>
__device__ __forceinline__ Tile tile_of(int u, const GemmParams& p, const SmemMeta& m, int n_sh_tiles, int mt_sh) {
    Tile tl;
    if (u < n_sh_tiles) {
        tl.prob = 1;
        tl.g = 0;
        tl.nt = u / mt_sh;
        const int mt = u % mt_sh;
        tl.row0 = mt * BM;
        tl.rows_valid = (int)min((int64_t)BM, p.T_sh - (int64_t)mt * BM);
        return tl;
    }
    u -= n_sh_tiles;
    int lo = 0, hi = p.G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (m.ts[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    const int g = lo;
    const int local = u - m.ts[g];
    const int M = m.off[g + 1] - m.off[g];
    const int MT = (M + BM - 1) / BM;
    tl.prob = 0;
    tl.g = g;
    tl.nt = local / MT;
    const int mt = local % MT;
    tl.row0 = m.off[g] + mt * BM;
    tl.rows_valid = min(BM, M - mt * BM);
    return tl;
}

template <bool kFC1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmAs,
                        const __grid_constant__ CUtensorMap tmBs) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* smA = smem;
    uint8_t* smB = smem + (size_t)STAGES * A_BYTES;
    SmemMeta& m = *reinterpret_cast<SmemMeta*>(smem + (size_t)STAGES * STAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int OW = kFC1 ? BN / 2 : BN;

    // ---------------- prologue ----------------
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.tfull[b], 1);
            mbar_init(&m.tempty[b], 4);
        }
        mbar_init(&m.drain, 1);
        m.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmAs);
        tma_prefetch_desc(&tmBs);
    }
    if (warp == 1) {
        tmem_alloc(&m.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) {
        // routed tile prefix: ts[g] = NT * sum_{g' < g} ceil(M_g' / BM)
        const int G = p.G;
        const int NT = (p.N_out + OW - 1) / OW;
        for (int i = lane; i <= G; i += 32) m.off[i] = (G > 0) ? p.offsets[i] : 0;
        __syncwarp();
        bool ok = true;
        for (int i = lane; i < G; i += 32) ok = ok && (m.off[i + 1] >= m.off[i]);
        if (lane == 0) ok = ok && (m.off[0] >= 0) && ((int64_t)m.off[G] <= p.rows_cap);
        ok = __all_sync(0xffffffffu, ok);
        const int C = (G + 31) / 32;
        const int beg = min(G, lane * C), end = min(G, beg + C);
        int local = 0;
        if (ok)
            for (int g = beg; g < end; ++g) local += ((m.off[g + 1] - m.off[g] + BM - 1) / BM) * NT;
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - local;
        for (int g = beg; g < end; ++g) {
            m.ts[g] = run;
            if (ok) run += ((m.off[g + 1] - m.off[g] + BM - 1) / BM) * NT;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) {
            m.ts[G] = total;
            m.routed_tiles = total;
            if (!ok) report(p.status, MOE_ERR_DEVICE_BOUNDS);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = m.tmem_base;
    const int mt_sh = p.T_sh > 0 ? (int)((p.T_sh + BM - 1) / BM) : 0;
    const int n_sh_tiles = p.T_sh > 0 ? mt_sh * ((p.N_out_sh + OW - 1) / OW) : 0;
    const int total_tiles = n_sh_tiles + m.routed_tiles;
    const volatile int* abortp = &m.abort;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool failed = false;
            for (int u = blockIdx.x; u < total_tiles && !failed; u += gridDim.x) {
                const Tile tl = tile_of<kFC1>(u, p, m, n_sh_tiles, mt_sh);
                const CUtensorMap* mA = tl.prob ? &tmAs : &tmA;
                const CUtensorMap* mB = tl.prob ? &tmBs : &tmB;
                const int nkb = (tl.prob ? p.K_sh : p.K) / BK;
                const int up = tl.prob ? p.up_off_sh : p.up_off;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&m.empty[stage], phase ^ 1u, p.timeout_ns, abortp)) {
                        failed = true;
                        break;
                    }
                    mbar_arrive_expect_tx(&m.full[stage], STAGE_BYTES);
                    uint8_t* a_dst = smA + (size_t)stage * A_BYTES;
                    uint8_t* b_dst = smB + (size_t)stage * B_BYTES;
                    tma_load_2d(a_dst, mA, &m.full[stage], kb * BK, tl.row0);
                    if (kFC1) {
                        tma_load_3d(b_dst, mB, &m.full[stage], kb * BK, tl.nt * (BN / 2), tl.g);
                        tma_load_3d(b_dst + B_BYTES / 2, mB, &m.full[stage], kb * BK, up + tl.nt * (BN / 2), tl.g);
                    } else {
                        tma_load_3d(b_dst, mB, &m.full[stage], kb * BK, tl.nt * BN, tl.g);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (failed) {
                m.abort = 1;
                report(p.status, MOE_ERR_TIMEOUT);
                // let the copies still in flight land before the CTA may exit
                for (int64_t j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j)
                    (void)mbar_wait(&m.full[j % STAGES], (uint32_t)((j / STAGES) & 1), p.timeout_ns, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            uint32_t stage = 0, phase = 0;
            bool failed = false;
            int i = 0;
            for (int u = blockIdx.x; u < total_tiles && !failed; u += gridDim.x, ++i) {
                const Tile tl = tile_of<kFC1>(u, p, m, n_sh_tiles, mt_sh);
                const int nkb = (tl.prob ? p.K_sh : p.K) / BK;
                const int buf = i & 1;
                if (!mbar_wait(&m.tempty[buf], (uint32_t)(((i >> 1) & 1) ^ 1), p.timeout_ns, abortp)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * BN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&m.full[stage], phase, p.timeout_ns, abortp)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smA + (size_t)stage * A_BYTES);
                    const uint32_t b0 = smem_u32(smB + (size_t)stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        tc_mma_bf16(d, sw128_kmajor_desc(a0 + kk * UMMA_K * 2), sw128_kmajor_desc(b0 + kk * UMMA_K * 2),
                                    IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(&m.empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (failed) break;
                tc_commit(&m.tfull[buf]);
            }
            if (failed) {
                m.abort = 1;
                report(p.status, MOE_ERR_TIMEOUT);
            }
            // all MMAs issued by this thread complete before TMEM is freed
            tc_commit(&m.drain);
            (void)mbar_wait(&m.drain, 0, p.timeout_ns, nullptr);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const int row_in = q * 32 + lane;    // tile row of this thread
        int i = 0;
        for (int u = blockIdx.x; u < total_tiles; u += gridDim.x, ++i) {
            const Tile tl = tile_of<kFC1>(u, p, m, n_sh_tiles, mt_sh);
            const int buf = i & 1;
            // every lane polls; the warp proceeds (reconverged, as tcgen05.ld
            // .sync.aligned requires) only if all lanes saw the phase complete
            const bool seen = mbar_wait(&m.tfull[buf], (uint32_t)((i >> 1) & 1), p.timeout_ns, abortp);
            if (!__all_sync(0xffffffffu, seen)) {
                if (lane == 0) {
                    m.abort = 1;
                    report(p.status, MOE_ERR_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(buf * BN) + ((uint32_t)(q * 32) << 16);
            const bool valid = row_in < tl.rows_valid;
            const int N_out = tl.prob ? p.N_out_sh : p.N_out;
            uint16_t* out = tl.prob ? p.out_sh : p.out;
            uint16_t* orow = out + (int64_t)(tl.row0 + row_in) * N_out;
            if (kFC1) {
#pragma unroll 1
                for (int c = 0; c < OW; c += 32) {
                    uint32_t g[32], v[32];
                    tmem_ld32(taddr + (uint32_t)c, g);
                    tmem_ld32(taddr + (uint32_t)(BN / 2 + c), v);
                    tmem_ld_wait();
                    const int col = tl.nt * OW + c;
                    if (valid && col < N_out) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float h2[2];
#pragma unroll
                            for (int z = 0; z < 2; ++z) {
                                const float gv = __uint_as_float(g[2 * e + z]);
                                const float uv = __uint_as_float(v[2 * e + z]);
                                // silu(g) * u; the product is rounded to bf16 (8 bits),
                                // far coarser than the approximate exp / divide
                                h2[z] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            }
                            pk[e] = pack_bf16x2(h2[0], h2[1]);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < OW; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)c, r);
                    tmem_ld_wait();
                    const int col = tl.nt * OW + c;
                    if (valid && col < N_out) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                        uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&m.tempty[buf]);
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

__global__ void wait_probe_kernel(int32_t* status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing ever arrives on `bar`: phase 0 never completes
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, timeout_ns, nullptr)) report(status, MOE_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t groups,
               uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, groups};
    cuuint64_t strides[2] = {inner * 2, rows * inner * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise the dynamic shared-memory limit of a kernel instantiation once per device.
template <bool kFC1>
cudaError_t configure_once() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kFC1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)SMEM_BYTES);
    if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return err;
}

}  // namespace

cudaError_t launch_grouped_gemm(const GemmLaunch& L, int num_sms, cudaStream_t s, const char** why) {
    const bool has_routed = L.G > 0 && L.rows_cap > 0;
    const bool has_shared = L.T_sh > 0 && L.b_sh != nullptr && L.N_out_sh > 0;
    if (!has_routed && !has_shared) return cudaSuccess;
    if (L.G > MAX_GROUPS) {
        *why = "too many groups";
        return cudaErrorInvalidValue;
    }
    const uint32_t brows = L.swiglu ? BN / 2 : BN;
    CUtensorMap mA, mB, mAs, mBs;
    bool ok = true;
    if (has_routed) {
        ok = ok && encode_2d(&mA, L.a, (uint64_t)L.K, (uint64_t)L.rows_cap, BM);
        ok = ok && encode_3d(&mB, L.b, (uint64_t)L.K, (uint64_t)L.Nb, (uint64_t)L.G, brows);
    }
    if (has_shared) {
        ok = ok && encode_2d(&mAs, L.a_sh, (uint64_t)L.K_sh, (uint64_t)L.T_sh, BM);
        ok = ok && encode_3d(&mBs, L.b_sh, (uint64_t)L.K_sh, (uint64_t)L.Nb_sh, 1, brows);
    }
    if (!ok) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    if (!has_routed) {
        mA = mAs;
        mB = mBs;
    }
    if (!has_shared) {
        mAs = mA;
        mBs = mB;
    }
    GemmParams p;
    p.offsets = L.offsets;
    p.G = has_routed ? L.G : 0;
    p.K = L.K;
    p.K_sh = L.K_sh;
    p.N_out = L.N_out;
    p.N_out_sh = L.N_out_sh;
    p.up_off = L.swiglu ? L.Nb / 2 : 0;
    p.up_off_sh = L.swiglu ? L.Nb_sh / 2 : 0;
    p.rows_cap = L.rows_cap;
    p.T_sh = has_shared ? L.T_sh : 0;
    p.out = L.out;
    p.out_sh = L.out_sh;
    p.status = &L.hdr->status;
    p.timeout_ns = L.timeout_ns;

    const int ow = L.swiglu ? BN / 2 : BN;
    int64_t bound = 0;
    if (has_routed) bound += (int64_t)((L.N_out + ow - 1) / ow) * ((L.rows_cap + BM - 1) / BM + L.G);
    if (has_shared) bound += (int64_t)((L.N_out_sh + ow - 1) / ow) * ((L.T_sh + BM - 1) / BM);
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(bound, num_sms));

    cudaError_t err = L.swiglu ? configure_once<true>() : configure_once<false>();
    if (err != cudaSuccess) {
        *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
        return err;
    }
    if (L.swiglu)
        grouped_gemm_kernel<true><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(p, mA, mB, mAs, mBs);
    else
        grouped_gemm_kernel<false><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(p, mA, mB, mAs, mBs);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(WsHeader* hdr, uint64_t timeout_ns, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(&hdr->status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace moe
