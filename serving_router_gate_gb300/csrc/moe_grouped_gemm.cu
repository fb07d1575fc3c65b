// moe_grouped_gemm.cu -- grouped GEMMs of the MoE experts on the tcgen05
// tensor cores (sm_103a): FC1 with a fused SwiGLU epilogue, and FC2.
//
// Method: per expert slot, the gated MLP (SwiGLU) of the TensorRT-LLM
// AutoDeploy MoE ops (PR #10985, "MoE all-to-all paradigm": is_gated_mlp and
// act_fn per expert); slots with no rows get no tiles (vLLM EP FusedMoE patch,
// module docstring: the per-expert loop skips experts with count 0).
//
// Design (persistent, one CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] (bf16,
//               128-byte swizzle) per K step into a 4-stage shared-memory ring;
//               a tile with at most 32 rows of its group loads only 32 A rows
//               (the MMA reads all 128; the rest are never stored).
//               FC1's B tile is two 128-row halves -- gate rows n0.. and up
//               rows I+n0.. -- so one MMA of N = 256 yields matching gate and
//               up columns, with no weight re-layout.
//   warp 1      tensor memory allocator (512 columns = 2 accumulators of
//               256 fp32 columns) and, on one thread, the MMA issuer:
//               tcgen05.mma.cta_group::1.kind::f16 M=128 N=256 K=16, four per
//               K step, completion signalled through tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31 = tile rows), FC1: h = bf16(silu(gate) * up);
//               FC2: y = bf16(acc); 16-byte stores (a routed row through the
//               caller's row map when one is given); rows past the slot's count
//               are not stored.  Two accumulators let the epilogue of one tile
//               overlap the main loop of the next.
// Pair mode (kPair, clusters of 2 CTAs): one tcgen05.mma.cta_group::2 of
// M = 256 spans the pair.  Each CTA stages its own 128 rows of A and one
// 128-row half of the B tile (32 KB per stage instead of 48, 6 stages), so every
// weight byte is read once per pair and each SM's shared memory carries half of
// B.  The leader (rank 0) issues the MMAs; both CTAs' copies are counted on the
// leader's stage barriers, its commits are multicast to both CTAs, and both
// CTAs' epilogues release the leader's accumulator barriers.  The two CTAs take
// consecutive m-tiles of one (slot, n-tile); an odd leftover m-tile leaves the
// second CTA without rows (its half is computed and discarded).  Single mode
// (one CTA per tile, 4 stages of 48 KB) serves small launches.
// E4M3 weights (quant GEMM_W8): 8 more warps widen each E4M3 weight tile to bf16
// in shared memory before the MMA reads it.  E4M3 weights and activations
// (GEMM_W8A8): the TMA loads 128-byte rows of E4M3 bytes (128 elements per K
// step instead of 64, same bytes per stage), tcgen05.mma.kind::f8f6f4 (K = 32)
// consumes them directly, and the epilogue scales each accumulator by its A
// row's and its B row's scale.
// Tiles: an optional dense "shared expert" problem (M = T) first, then the
// routed problem, whose ragged per-slot row counts are read on the device from
// the offsets array (no host synchronisation): slot g has ceil(M_g / 128)
// m-tiles; within a slot, tiles run n-tile-major so consecutive CTAs share the
// same weight tile through L2.  The CTAs take tiles round-robin; when the shared
// tiles are longer than the routed ones, a CTA with one shared tile fewer first
// takes as many routed tiles as make up the difference.  The shared tiles start
// before the routed prefix is built (it arrives on an mbarrier).  Every wait is
// bounded: on a timeout the CTA
// records MOE_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees its
// tensor memory and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 128;            // rows of A per CTA
constexpr int BK = 64;             // bf16 elements per 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;
constexpr int BM_SHORT = 32;                      // A rows loaded for tiles with at most 32 rows
constexpr int A_SHORT_BYTES = BM_SHORT * BK * 2;
constexpr int NUM_THREADS = 192;
constexpr int NUM_THREADS_FP8 = 448;  // plus warps 6..13: E4M3 -> bf16 converters
constexpr int NUM_THREADS_F4 = 256;   // plus warps 6..7: NVFP4 block-scale layout converters
constexpr int F4_CONV_THREADS = 64;
constexpr int SF_STAGE_BYTES = 4096;  // NVFP4: the A and the B block scales of a stage, 2 KB each
constexpr int CONV_THREADS = 256;
constexpr int CONV_BARRIER = 1;       // named barrier of the converter warps
constexpr int MAX_GROUPS = 1024;
constexpr int MAX_STAGES = 8;
constexpr int RING_BYTES = 216 * 1024;  // shared memory for the operand ring
constexpr uint16_t PAIR_MASK = 0x3;

// per instantiation: MMA N = BN (256 for large launches, 128 / 64 to spread
// small ones over more CTAs); a CTA holds all of B (single) or its half (pair).
// A stage holds KS consecutive K chunks of 64 bf16 (one 128-byte swizzle row per
// operand row each): chunk c of A at c * A_CHUNK, of B at c * B_CHUNK.
template <bool kPair, int BN, bool kShort = false, int KS = 1, int SFB = 0>
struct Cfg {
    static constexpr int B_CHUNK = (kPair ? BN / 2 : BN) * BK * 2;
    static constexpr int B_BYTES = B_CHUNK * KS;
    // kShort: every tile has at most 32 rows, so an A slot holds 32 rows per chunk (the
    // MMA still reads 128 rows from the chunk onward; rows past 32 are never stored)
    static constexpr int A_CHUNK = kShort ? A_SHORT_BYTES : A_BYTES;
    static constexpr int A_SLOT = A_CHUNK * KS;
    static constexpr int STAGE_BYTES = A_SLOT + B_BYTES + SFB;  // SFB: NVFP4 block scales
    static constexpr int STAGES = RING_BYTES / STAGE_BYTES < MAX_STAGES ? RING_BYTES / STAGE_BYTES : MAX_STAGES;
    static constexpr int TMEM_COLS = 2 * BN;  // two accumulators of BN fp32 columns
    // 2-CTA MMA: M = 256 across the pair
    static constexpr uint32_t IDESC = idesc_bf16_f32(kPair ? 2 * BM : BM, BN);
};

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
    const int32_t* out_row;  // or [rows_cap]: routed row r is stored at out row out_row[r]
    const float* scale;      // E4M3 weights: fp32 scale per B row, [G][Nb] (null: bf16 weights)
    const float* scale_sh;   // [Nb_sh]
    const float* a_scale;    // E4M3 activations: fp32 scale per A row, [rows_cap]
    const float* a_scale_sh; // [T_sh]
    int kb_total, kb_total_sh;  // K steps of the routed and the shared problem
    int Nb;                  // B rows per group
    float* out_sh_part;      // FC2, split shared problem: fp32 partials [ksplit_sh, T_sh, N_out_sh]
    int ksplit_sh;           // K ranges of the shared problem (1: not split)
    int kb_split_sh;         // K steps per range
    int prefetch_sh;         // FC1: pull this CTA's shared-problem weights into L2 before
                             // waiting on the previous kernel (shared problems of <= 64 rows)
    int32_t* status;
    uint64_t timeout_ns;
};

struct SmemMeta {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t conv[MAX_STAGES];  // E4M3 weights: stage converted to bf16 (8 converter warps)
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t ready;   // the routed tile prefix (off, ts, routed_tiles) is written
    uint32_t tmem_base;
    int abort;
    volatile int conv_ok;
    int routed_tiles;
    int off[MAX_GROUPS + 1];
    int ts[MAX_GROUPS + 1];
};

// K chunks per stage: two for short-tile (small-batch) bf16 launches, whose CTAs
// stream weights at a pace set by the number of pipeline stages they issue, not by
// the bytes; one otherwise
template <bool kShort, int kQ>
constexpr int chunks_per_stage() {
    return (kShort && kQ == 0) ? 2 : 1;
}

// block-scale bytes of a pipeline stage
template <int kQ>
constexpr int sf_stage_bytes() {
    return kQ == GEMM_NVFP4 ? SF_STAGE_BYTES : 0;
}

template <int kQ>
constexpr int threads_of() {
    return kQ == GEMM_W8 ? NUM_THREADS_FP8 : (kQ == GEMM_NVFP4 ? NUM_THREADS_F4 : NUM_THREADS);
}

template <bool kPair, int BN, bool kShort, int KS, int SFB>
constexpr size_t smem_bytes() {
    return 1024 /*alignment slack*/ +
           (size_t)Cfg<kPair, BN, kShort, KS, SFB>::STAGES * Cfg<kPair, BN, kShort, KS, SFB>::STAGE_BYTES +
           sizeof(SmemMeta);
}

struct Tile {
    int prob;        // 0 routed, 1 shared
    int g;           // routed group
    int nt;          // n-tile
    int row0;        // first row in A / out of this CTA's m-tile
    int rows_valid;  // rows of this CTA's m-tile that belong to the group (may be 0)
    int ks;          // K range of a split shared tile (0 otherwise)
    int kb0, kb1;    // K steps [kb0, kb1) of this tile
};

// work units along M: pairs of m-tiles in pair mode, single m-tiles otherwise
template <bool kPair>
__device__ __forceinline__ int units_of(int mtiles) {
    return kPair ? (mtiles + 1) >> 1 : mtiles;
}

template <bool kFC1, bool kPair>
__device__ __forceinline__ Tile tile_of(int u, const GemmParams& p, const SmemMeta& m, int n_sh_tiles, int mu_sh,
                                        int crank) {
    Tile tl;
    if (u < n_sh_tiles) {
        // split shared tiles: the K ranges of one output tile are consecutive units
        tl.prob = 1;
        tl.g = 0;
        tl.ks = u % p.ksplit_sh;
        const int v = u / p.ksplit_sh;
        tl.nt = v / mu_sh;
        const int mt = kPair ? 2 * (v % mu_sh) + crank : v % mu_sh;
        tl.row0 = mt * BM;
        tl.rows_valid = (int)max((int64_t)0, min((int64_t)BM, p.T_sh - (int64_t)mt * BM));
        tl.kb0 = tl.ks * p.kb_split_sh;
        tl.kb1 = min(p.kb_total_sh, tl.kb0 + p.kb_split_sh);
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
    const int MU = units_of<kPair>((M + BM - 1) / BM);
    tl.prob = 0;
    tl.g = g;
    tl.nt = local / MU;
    const int mt = kPair ? 2 * (local % MU) + crank : local % MU;
    tl.row0 = m.off[g] + mt * BM;
    tl.rows_valid = max(0, min(BM, M - mt * BM));
    tl.ks = 0;
    tl.kb0 = 0;
    tl.kb1 = p.kb_total;
    return tl;
}

// Four E4M3 weights (one 32-bit word) -> four bf16 values (two words), exactly,
// with integer operations on two 16-bit halves at a time.  A normal E4M3 value
// (exponent field e >= 1) keeps its mantissa and gets the exponent
// e - 7 + 127: bf16 = (mag << 4) + (120 << 7), sign moved from bit 7 to bit 15.
// Zeros and subnormals (e = 0: m * 2^-9) are rare; a word holding one takes a
// slow path that places the byte's fields in binary32 positions and scales by
// 2^120 (exact, including binary32 subnormal inputs), keeping the top 16 bits.
__device__ __forceinline__ uint32_t e4m3_small_to_bf16(uint32_t mag) {
    return __float_as_uint(__uint_as_float(mag << 20) * 0x1p120f) >> 16;
}

__device__ __forceinline__ uint32_t e4m3x2_normal_to_bf16x2(uint32_t v) {  // bytes at bits 0-7 and 16-23
    return ((v & 0x007F007Fu) * 16u + 0x3C003C00u) | ((v << 8) & 0x80008000u);
}

__device__ __forceinline__ uint32_t e4m3x2_any_to_bf16x2(uint32_t v) {
    const uint32_t lo = v & 0x7Fu, hi = (v >> 16) & 0x7Fu;
    const uint32_t blo = (lo & 0x78u) ? lo * 16u + 0x3C00u : e4m3_small_to_bf16(lo);
    const uint32_t bhi = (hi & 0x78u) ? hi * 16u + 0x3C00u : e4m3_small_to_bf16(hi);
    return (blo | (bhi << 16)) | ((v << 8) & 0x80008000u);
}

__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t x, uint32_t& o0, uint32_t& o1) {
    const uint32_t a = __byte_perm(x, 0u, 0x4140), b = __byte_perm(x, 0u, 0x4342);  // bytes 0,1 and 2,3
    const uint32_t t = x & 0x78787878u;                                               // exponent fields
    if (((t - 0x08080808u) & ~t & 0x80808080u) == 0u) {  // no zero exponent field among the four
        o0 = e4m3x2_normal_to_bf16x2(a);
        o1 = e4m3x2_normal_to_bf16x2(b);
    } else {
        o0 = e4m3x2_any_to_bf16x2(a);
        o1 = e4m3x2_any_to_bf16x2(b);
    }
}

template <bool kFC1, bool kPair, int BN, bool kShort, int kQ>
__global__ void __launch_bounds__(threads_of<kQ>(), 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmAs,
                        const __grid_constant__ CUtensorMap tmBs, const __grid_constant__ CUtensorMap tmA32,
                        const __grid_constant__ CUtensorMap tmAs32, const __grid_constant__ CUtensorMap tmSFA,
                        const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmSFAs,
                        const __grid_constant__ CUtensorMap tmSFBs) {
    constexpr int KSC = chunks_per_stage<kShort, kQ>();
    using C = Cfg<kPair, BN, kShort, KSC, sf_stage_bytes<kQ>()>;
    constexpr int STAGES = C::STAGES;
    constexpr int B_BYTES = C::B_BYTES;
    constexpr int A_SLOT = C::A_SLOT;
    constexpr uint32_t IDESC = C::IDESC;
    constexpr uint32_t IDESC4 = idesc_nvfp4(BM, BN);
    constexpr int TMEM_COLS = C::TMEM_COLS;
    static_assert(!kShort || !kPair, "short tiles run in single mode");
    constexpr bool kFp8 = kQ == GEMM_W8;      // E4M3 weights widened by converter warps
    constexpr bool kA8 = kQ == GEMM_W8A8;     // E4M3 A and B on kind::f8f6f4
    constexpr bool kF4 = kQ == GEMM_NVFP4;    // E2M1 A and B with E4M3 block scales on kind::mxf4nvf4
    constexpr int KE = kF4 ? 4 * BK : (kA8 ? 2 * BK : BK);  // elements per K step (one 128-byte row)
    // NVFP4: two accumulators, then two sets (stage parity) of 32 block-scale columns
    constexpr int TMEM_ALLOC = kF4 ? 512 : TMEM_COLS;
    static_assert(!kF4 || (!kPair && BN == 128 && 2 * BN + 64 <= TMEM_ALLOC), "NVFP4 runs single CTAs with N = 128");
    static_assert(!kFp8 || (!kPair && BN == 256), "E4M3 weights run in single mode with N = 256");
    static_assert(!kA8 || !kPair, "E4M3 activations run in single mode");
    static_assert(!kPair || BN == 256, "pair mode uses N = 256");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* smA = smem;
    uint8_t* smB = smem + (size_t)STAGES * A_SLOT;
    uint8_t* smSF = smB + (size_t)STAGES * B_BYTES;  // NVFP4: [stage][A scales 2 KB][B scales 2 KB]
    SmemMeta& m = *reinterpret_cast<SmemMeta*>(smem + (size_t)STAGES * C::STAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int OW = kFC1 ? BN / 2 : BN;
    const int crank = kPair ? (int)cluster_ctarank() : 0;
    const int unit0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nunits = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    // ---------------- prologue ----------------
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&m.full[s], 1);   // pair mode: only the leader's, fed by both CTAs' copies
            mbar_init(&m.empty[s], 1);  // released by the (leader's) MMA commit
            if (kFp8) mbar_init(&m.conv[s], CONV_THREADS / 32);  // one arrival per converter warp
            if (kF4) mbar_init(&m.conv[s], F4_CONV_THREADS / 32);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.tfull[b], 1);
            mbar_init(&m.tempty[b], kPair ? 8 : 4);  // pair mode: the epilogue warps of both CTAs
        }
        mbar_init(&m.drain, 1);
        mbar_init(&m.ready, 1);
        m.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmAs);
        tma_prefetch_desc(&tmBs);
        tma_prefetch_desc(&tmA32);
        tma_prefetch_desc(&tmAs32);
        if (kF4) {
            tma_prefetch_desc(&tmSFA);
            tma_prefetch_desc(&tmSFB);
            tma_prefetch_desc(&tmSFAs);
            tma_prefetch_desc(&tmSFBs);
        }
    }
    if (warp == 1) {
        if (kPair) {
            tmem_alloc_pair(&m.tmem_base, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&m.tmem_base, TMEM_ALLOC);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if (kPair) {
        __syncwarp();        // barrier.cluster.*.aligned: each warp arrives converged
        cluster_sync_all();  // the peer's multicasts may target this CTA's barriers from here on
    } else {
        __syncthreads();
    }
    tc_fence_after();

    const uint32_t tmem_base = m.tmem_base;
    const int mu_sh = p.T_sh > 0 ? units_of<kPair>((int)((p.T_sh + BM - 1) / BM)) : 0;
    const int n_sh_tiles = p.T_sh > 0 ? mu_sh * ((p.N_out_sh + OW - 1) / OW) * p.ksplit_sh : 0;
    const volatile int* abortp = &m.abort;
    // This CTA's units, in order: its shared-problem units unit0 + j * nunits first
    // (they need no prefix), then routed units, once m.ready has published the prefix.
    // Where the shared units split unevenly over the CTAs, each CTA with one shared unit
    // fewer first takes q routed units (q = the shared-to-routed K-step ratio, rounded),
    // so the K steps per CTA even out; the remaining routed units go round-robin.  With
    // q = 1, or fewer than q routed units per CTA (streaming launches, where spreading
    // the units over more SMs matters more), this is plain round-robin over all units.  next_unit(i) returns the
    // i-th unit, -1 past the last, -2 if the wait for the prefix gave up.
    const int n_long = unit0 < n_sh_tiles ? (n_sh_tiles - unit0 + nunits - 1) / nunits : 0;
    const int light0 = n_sh_tiles % nunits;  // first CTA with one shared unit fewer
    const int len_sh = p.ksplit_sh > 1 ? p.kb_split_sh : p.kb_total_sh;
    const int len_rt = max(1, p.kb_total);
    const int bonus_q = light0 == 0 ? 0 : max(1, (len_sh + len_rt / 2) / len_rt);
    auto next_unit = [&](int i, bool& have) -> int {
        if (i < n_long) return unit0 + i * nunits;
        if (!have) {
            if (!mbar_wait(&m.ready, 0, p.timeout_ns, abortp)) return -2;
            have = true;
        }
        const int routed = m.routed_tiles;
        int j = i - n_long;
        int bonus_total = 0;
        if (bonus_q > 0) {
            const int q = routed >= nunits * bonus_q ? bonus_q : 1;
            bonus_total = min((nunits - light0) * q, routed);
            if (unit0 >= light0) {
                const int b0 = (unit0 - light0) * q;
                const int nb = max(0, min(q, bonus_total - b0));
                if (j < nb) return n_sh_tiles + b0 + j;
                j -= nb;
            }
        }
        const int r = bonus_total + unit0 + j * nunits;
        return r < routed ? n_sh_tiles + r : -1;
    };

    // FC1 with a shared problem of few rows reads each shared weight byte once, and the
    // weights are no earlier kernel's output: an idle epilogue warp pulls this CTA's shared
    // tiles of them into L2 while the previous kernel on the stream (the permutation) still
    // runs, so the shared expert's HBM stream overlaps the routing kernels.  (Without
    // programmatic launch the wait below returns at once and the prefetch just leads the
    // loads.)
    if constexpr (kFC1 && !kPair) {
        if (p.prefetch_sh && warp == 3 && lane == 0) {
            for (int i = 0; i < n_long; ++i) {
                const Tile tl = tile_of<kFC1, kPair>(unit0 + i * nunits, p, m, n_sh_tiles, mu_sh, crank);
                for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                    const int kx = kF4 ? kb * 128 : kb * KE;  // x in bytes: packed E2M1 holds two per byte
                    tma_prefetch_l2_3d(&tmBs, kx, tl.nt * (BN / 2), 0);
                    tma_prefetch_l2_3d(&tmBs, kx, p.up_off_sh + tl.nt * (BN / 2), 0);
                }
            }
        }
    }

    // everything above touches no memory of earlier kernels; from here on it may.
    // The shared problem's units need only their operands, so the roles start on
    // them at once; warp 2 meanwhile builds the routed tile prefix from the offsets
    // and publishes it on m.ready, which every role waits for before its first
    // routed unit.
    pdl_wait();
    pdl_trigger();
    if (warp == 2) {
        // routed unit prefix: ts[g] = NT * sum_{g' < g} units(ceil(M_g' / BM))
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
            for (int g = beg; g < end; ++g) local += units_of<kPair>((m.off[g + 1] - m.off[g] + BM - 1) / BM) * NT;
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - local;
        for (int g = beg; g < end; ++g) {
            m.ts[g] = run;
            if (ok) run += units_of<kPair>((m.off[g + 1] - m.off[g] + BM - 1) / BM) * NT;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) {
            m.ts[G] = total;
            m.routed_tiles = total;
            if (!ok) report(p.status, MOE_ERR_DEVICE_BOUNDS);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.ready);
    }

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool failed = false;
            bool have = false;
            for (int iu = 0; !failed; ++iu) {
                const int u = next_unit(iu, have);
                if (u == -2) {
                    failed = true;
                    break;
                }
                if (u < 0) break;
                const Tile tl = tile_of<kFC1, kPair>(u, p, m, n_sh_tiles, mu_sh, crank);
                // a tile with at most 32 rows of its group loads only 32 A rows: the MMA
                // still reads 128, but rows past the group's count are never stored
                const bool short_a = kShort || tl.rows_valid <= BM_SHORT;
                const CUtensorMap* mA = tl.prob ? (short_a ? &tmAs32 : &tmAs) : (short_a ? &tmA32 : &tmA);
                const CUtensorMap* mB = tl.prob ? &tmBs : &tmB;
                const int up = tl.prob ? p.up_off_sh : p.up_off;
                const uint32_t a_bytes = short_a ? A_SHORT_BYTES : A_BYTES;
                uint32_t pair_bytes = 0;  // pair mode: bytes of both CTAs, counted by the leader
                if (kPair) {
                    const Tile other = tile_of<kFC1, kPair>(u, p, m, n_sh_tiles, mu_sh, crank ^ 1);
                    pair_bytes = a_bytes + (other.rows_valid <= BM_SHORT ? A_SHORT_BYTES : A_BYTES) + 2 * B_BYTES;
                }
                for (int kb = tl.kb0; kb < tl.kb1; kb += KSC) {
                    if (!mbar_wait(&m.empty[stage], phase ^ 1u, p.timeout_ns, abortp)) {
                        failed = true;
                        break;
                    }
                    uint8_t* a_dst = smA + (size_t)stage * A_SLOT;
                    uint8_t* b_dst = smB + (size_t)stage * B_BYTES;
                    if (kPair) {
                        // this CTA's A rows and its 128-row half of B; the bytes of both
                        // CTAs are counted on the leader's stage barrier
                        const uint32_t lead_full = mapa_shared(&m.full[stage], 0);
                        if (crank == 0) mbar_arrive_expect_tx(&m.full[stage], pair_bytes);
                        const int brow = kFC1 ? (crank ? up : 0) + tl.nt * (BN / 2) : tl.nt * BN + crank * (BN / 2);
                        tma_load_2d_pair(a_dst, mA, lead_full, kb * KE, tl.row0);
                        tma_load_3d_pair(b_dst, mB, lead_full, kb * KE, brow, tl.g);
                    } else if (kFp8) {
                        // E4M3 rows of 64 bytes, dense, in the first half of the B slot (FC1:
                        // the gate rows, then the up rows); the converters widen them in place
                        mbar_arrive_expect_tx(&m.full[stage], a_bytes + BN * BK);
                        tma_load_2d(a_dst, mA, &m.full[stage], kb * KE, tl.row0);
                        if (kFC1) {
                            tma_load_3d(b_dst, mB, &m.full[stage], kb * KE, tl.nt * (BN / 2), tl.g);
                            tma_load_3d(b_dst + (BN / 2) * BK, mB, &m.full[stage], kb * KE, up + tl.nt * (BN / 2), tl.g);
                        } else {
                            tma_load_3d(b_dst, mB, &m.full[stage], kb * KE, tl.nt * BN, tl.g);
                        }
                    } else if (kF4) {
                        // 128-byte rows of packed E2M1 codes (256 elements) and, for the same
                        // 256 elements, 16 bytes of block scales per row: A's tile rows from
                        // row0, B's rows as the codes (FC1: gate rows, then up rows)
                        const CUtensorMap* mSA = tl.prob ? &tmSFAs : &tmSFA;
                        const CUtensorMap* mSB = tl.prob ? &tmSFBs : &tmSFB;
                        constexpr uint32_t SFA_BOX = (kShort ? BM_SHORT : BM) * 16;
                        mbar_arrive_expect_tx(&m.full[stage], a_bytes + B_BYTES + SFA_BOX + BN * 16);
                        const int kx = kb * 128, ks = kb * 16;
                        uint8_t* sfa = smSF + (size_t)stage * SF_STAGE_BYTES;
                        uint8_t* sfb = sfa + SF_STAGE_BYTES / 2;
                        tma_load_2d(a_dst, mA, &m.full[stage], kx, tl.row0);
                        tma_load_3d(sfa, mSA, &m.full[stage], ks, tl.row0, 0);
                        if (kFC1) {
                            tma_load_3d(b_dst, mB, &m.full[stage], kx, tl.nt * (BN / 2), tl.g);
                            tma_load_3d(b_dst + B_BYTES / 2, mB, &m.full[stage], kx, up + tl.nt * (BN / 2), tl.g);
                            tma_load_3d(sfb, mSB, &m.full[stage], ks, tl.nt * (BN / 2), tl.g);
                            tma_load_3d(sfb + (BN / 2) * 16, mSB, &m.full[stage], ks, up + tl.nt * (BN / 2), tl.g);
                        } else {
                            tma_load_3d(b_dst, mB, &m.full[stage], kx, tl.nt * BN, tl.g);
                            tma_load_3d(sfb, mSB, &m.full[stage], ks, tl.nt * BN, tl.g);
                        }
                    } else {
                        // KSC chunks: a chunk past the range's end lies past K (ranges of
                        // split tiles are multiples of KSC), where the TMA fills zeros
                        mbar_arrive_expect_tx(&m.full[stage], KSC * (a_bytes + C::B_CHUNK));
#pragma unroll
                        for (int c = 0; c < KSC; ++c) {
                            const int kc = (kb + c) * KE;
                            tma_load_2d(a_dst + c * C::A_CHUNK, mA, &m.full[stage], kc, tl.row0);
                            uint8_t* bc = b_dst + c * C::B_CHUNK;
                            if (kFC1) {
                                tma_load_3d(bc, mB, &m.full[stage], kc, tl.nt * (BN / 2), tl.g);
                                tma_load_3d(bc + C::B_CHUNK / 2, mB, &m.full[stage], kc, up + tl.nt * (BN / 2), tl.g);
                            } else {
                                tma_load_3d(bc, mB, &m.full[stage], kc, tl.nt * BN, tl.g);
                            }
                        }
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
                // let the copies still in flight land before the CTA may exit (in pair
                // mode both CTAs' copies complete on the leader's barriers)
                if (!kPair || crank == 0)
                    for (int64_t j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j)
                        (void)mbar_wait(&m.full[j % STAGES], (uint32_t)((j / STAGES) & 1), p.timeout_ns, nullptr);
            }
            // tail: wait until the MMAs have released the last stages, so no commit
            // arrival can target this CTA after it exits
            for (int j = 0; j < STAGES; ++j) {
                (void)mbar_wait(&m.empty[stage], phase ^ 1u, p.timeout_ns, nullptr);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && crank == 0) {
            // ---------------- MMA issuer (the pair's leader in pair mode) ----------------
            uint32_t stage = 0, phase = 0;
            uint32_t sfp = 0;  // NVFP4: block-scale columns of this stage (two sets, alternating)
            bool failed = false;
            int i = 0;
            bool have = false;
            for (;; ++i) {
                const int u = next_unit(i, have);
                if (u == -2) {
                    failed = true;
                    break;
                }
                if (u < 0) break;
                const Tile tl = tile_of<kFC1, kPair>(u, p, m, n_sh_tiles, mu_sh, crank);
                const int nkb = (tl.kb1 - tl.kb0 + KSC - 1) / KSC;  // stages of this tile
                const int buf = i & 1;
                if (!mbar_wait(&m.tempty[buf], (uint32_t)(((i >> 1) & 1) ^ 1), p.timeout_ns, abortp)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * BN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait((kFp8 || kF4) ? &m.conv[stage] : &m.full[stage], phase, p.timeout_ns, abortp)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smA + (size_t)stage * A_SLOT);
                    const uint32_t b0 = smem_u32(smB + (size_t)stage * B_BYTES);
                    if constexpr (kF4) {
                        // per MMA of 64 elements: the A and B block scales of its 4 blocks
                        // (laid out by the converter warps) into tensor memory, then the MMA
                        const uint32_t sf0 = smem_u32(smSF + (size_t)stage * SF_STAGE_BYTES);
                        const uint32_t col = tmem_base + (uint32_t)(2 * BN) + (sfp & 1u) * 32u;
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            tc_copy_32x128b_x4(col + kk * 4, sf0 + kk * 512);
                            tc_copy_32x128b_x4(col + 16 + kk * 4, sf0 + SF_STAGE_BYTES / 2 + kk * 512);
                            const uint64_t ad = sw128_kmajor_desc(a0 + kk * UMMA_K * 2);
                            const uint64_t bd = sw128_kmajor_desc(b0 + kk * UMMA_K * 2);
                            tc_mma_nvfp4(d, ad, bd, IDESC4, col + kk * 4, col + 16 + kk * 4, (kb | kk) != 0 ? 1u : 0u);
                        }
                        ++sfp;
                    } else {
#pragma unroll
                    for (int c = 0; c < KSC; ++c)
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            // 32 bytes of each 128-byte row per MMA: K = 16 bf16 or 32 E4M3
                            const uint64_t ad = sw128_kmajor_desc(a0 + c * C::A_CHUNK + kk * UMMA_K * 2);
                            const uint64_t bd = sw128_kmajor_desc(b0 + c * C::B_CHUNK + kk * UMMA_K * 2);
                            const uint32_t acc = (kb | c | kk) != 0 ? 1u : 0u;
                            if (kPair)
                                tc_mma_bf16_pair(d, ad, bd, IDESC, acc);
                            else if (kA8)
                                tc_mma_e4m3(d, ad, bd, idesc_e4m3_f32(BM, BN), acc);
                            else
                                tc_mma_bf16(d, ad, bd, IDESC, acc);
                        }
                    }
                    if (kPair)
                        tc_commit_pair_multicast(&m.empty[stage], PAIR_MASK);
                    else
                        tc_commit(&m.empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (failed) break;
                if (kPair)
                    tc_commit_pair_multicast(&m.tfull[buf], PAIR_MASK);
                else
                    tc_commit(&m.tfull[buf]);
            }
            if (failed) {
                m.abort = 1;
                report(p.status, MOE_ERR_TIMEOUT);
            }
            // all MMAs issued by this thread complete before TMEM is freed
            if (kPair)
                tc_commit_pair_multicast(&m.drain, 0x1);
            else
                tc_commit(&m.drain);
            (void)mbar_wait(&m.drain, 0, p.timeout_ns, nullptr);
        }
    } else if (warp >= 2 && warp <= 5) {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const int row_in = q * 32 + lane;    // tile row of this thread
        int i = 0;
        bool have = false;
        for (;; ++i) {
            // every lane waits; the warp goes on only if all of them saw the prefix
            const int u = next_unit(i, have);
            if (!__all_sync(0xffffffffu, u != -2)) {
                if (lane == 0) {
                    m.abort = 1;
                    report(p.status, MOE_ERR_TIMEOUT);
                }
                break;
            }
            if (u < 0) break;
            const Tile tl = tile_of<kFC1, kPair>(u, p, m, n_sh_tiles, mu_sh, crank);
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
            // short-tile launches hold 32 A rows: a taller tile (a caller's bound was
            // wrong) is reported and only its first 32 rows are stored
            if (kShort && tl.rows_valid > BM_SHORT && row_in == 0) report(p.status, MOE_ERR_DEVICE_BOUNDS);
            bool valid = row_in < (kShort ? min(tl.rows_valid, BM_SHORT) : tl.rows_valid) &&
                         in_bounds(tl.row0 + row_in, tl.prob ? p.T_sh : p.rows_cap, p.status);
            int64_t orow_i = (int64_t)tl.row0 + row_in;
            if (p.out_row && !tl.prob && valid) {  // routed rows stored through the caller's row map
                orow_i = __ldg(p.out_row + orow_i);
                valid = in_bounds(orow_i, p.rows_cap, p.status);
            }
            const int N_out = tl.prob ? p.N_out_sh : p.N_out;
            uint16_t* out = tl.prob ? p.out_sh : p.out;
            uint16_t* orow = out + orow_i * N_out;
            // E4M3 weights: the accumulator of output column n carries B row n's scale;
            // E4M3 activations: and its A row's scale (a power of two)
            constexpr bool kRowScaleB = kFp8 || kA8 || kF4, kRowScaleA = kA8 || kF4;
            const float* srow = kRowScaleB ? (tl.prob ? p.scale_sh : p.scale + (int64_t)tl.g * p.Nb) : nullptr;
            const int sup = tl.prob ? p.up_off_sh : p.up_off;
            const float asc =
                (kRowScaleA && valid) ? __ldg((tl.prob ? p.a_scale_sh : p.a_scale) + tl.row0 + row_in) : 1.0f;
            auto bscale = [&](int row) -> float { return kRowScaleB ? __ldg(srow + row) : 1.0f; };
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
                                const float gv = __uint_as_float(g[2 * e + z]) * bscale(col + 2 * e + z) * asc;
                                const float uv = __uint_as_float(v[2 * e + z]) * bscale(sup + col + 2 * e + z) * asc;
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
            } else if (tl.prob && p.ksplit_sh > 1) {
                // K range ks of a split shared tile: fp32 partial sums, added up in fixed
                // range order by the combine; a range past the last K step (more ranges
                // than K steps allow) issued no MMA and contributes zeros
                float* prow = p.out_sh_part + ((int64_t)tl.ks * p.T_sh + tl.row0 + row_in) * N_out;
                const float kz = tl.kb1 > tl.kb0 ? 1.0f : 0.0f;
#pragma unroll 1
                for (int c = 0; c < OW; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)c, r);
                    tmem_ld_wait();
                    const int col = tl.nt * OW + c;
                    if (valid && col < N_out) {
                        float4* dst = reinterpret_cast<float4*>(prow + col);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = kz == 0.0f
                                         ? make_float4(0.f, 0.f, 0.f, 0.f)
                                         : make_float4(__uint_as_float(r[4 * e]) * bscale(col + 4 * e) * asc,
                                                       __uint_as_float(r[4 * e + 1]) * bscale(col + 4 * e + 1) * asc,
                                                       __uint_as_float(r[4 * e + 2]) * bscale(col + 4 * e + 2) * asc,
                                                       __uint_as_float(r[4 * e + 3]) * bscale(col + 4 * e + 3) * asc);
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
                            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * bscale(col + 2 * e) * asc,
                                                __uint_as_float(r[2 * e + 1]) * bscale(col + 2 * e + 1) * asc);
                        uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kPair)
                    mbar_arrive_cluster(mapa_shared(&m.tempty[buf], 0));  // the leader's barrier
                else
                    mbar_arrive(&m.tempty[buf]);
            }
        }
    } else if (kFp8 && warp >= 6) {
        // ---------------- E4M3 -> bf16 converters (warps 6..13) ----------------
        // Per K step the B slot holds BN rows of 64 E4M3 bytes (dense); the 256
        // threads read all of it, meet at a named barrier, then write the rows back
        // as bf16 in the 128-byte-swizzled layout the MMA reads (16-byte chunk j of
        // row r at r * 128 + ((j ^ (r & 7)) << 4)), which covers the whole slot.
        const int ct = threadIdx.x - 6 * 32;  // 0 .. CONV_THREADS - 1
        constexpr int CPT = (BN * 4 + CONV_THREADS - 1) / CONV_THREADS;  // 16-byte E4M3 chunks per thread
        uint32_t stage = 0, phase = 0;
        bool failed = false;
        // the tile sequence of all units is needed up front (one thread waits for the
        // prefix; the named barrier passes its verdict on)
        if (ct == 0) m.conv_ok = mbar_wait(&m.ready, 0, p.timeout_ns, abortp) ? 1 : 0;
        asm volatile("bar.sync %0, %1;" ::"n"(CONV_BARRIER), "n"(CONV_THREADS) : "memory");
        failed = !m.conv_ok;
        bool have = true;  // the prefix is published (waited for above)
        for (int iu = 0; !failed; ++iu) {
            const int u = next_unit(iu, have);
            if (u < 0) break;
            const Tile tl = tile_of<kFC1, kPair>(u, p, m, n_sh_tiles, mu_sh, crank);
            const int nkb = tl.kb1 - tl.kb0;
            for (int kb = 0; kb < nkb; ++kb) {
                // one thread waits for the stage; the named barrier passes its verdict
                // (and, with it, the visibility of the landed bytes) to all of them, so
                // the warps always take the same branch and every barrier completes
                if (ct == 0) m.conv_ok = mbar_wait(&m.full[stage], phase, p.timeout_ns, abortp) ? 1 : 0;
                asm volatile("bar.sync %0, %1;" ::"n"(CONV_BARRIER), "n"(CONV_THREADS) : "memory");
                if (!m.conv_ok) {
                    failed = true;
                    break;
                }
                uint8_t* b_slot = smB + (size_t)stage * B_BYTES;
                // 16-byte chunk i of the slot's E4M3 rows (row i / 4, bytes 16 (i % 4) ..):
                // consecutive lanes read consecutive chunks (no bank conflicts)
                uint4 src[CPT];
#pragma unroll
                for (int j = 0; j < CPT; ++j)
                    src[j] = *reinterpret_cast<const uint4*>(b_slot + (size_t)(ct + j * CONV_THREADS) * 16);
                asm volatile("bar.sync %0, %1;" ::"n"(CONV_BARRIER), "n"(CONV_THREADS) : "memory");
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    const int i = ct + j * CONV_THREADS;
                    const int r = i >> 2, c = i & 3;
                    uint8_t* drow = b_slot + (size_t)r * 128;
                    const uint32_t w4[4] = {src[j].x, src[j].y, src[j].z, src[j].w};
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) e4m3x4_to_bf16x4(w4[e], o[2 * e], o[2 * e + 1]);
                    *reinterpret_cast<uint4*>(drow + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(drow + (((2 * c + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
                // generic-proxy stores -> visible to the tensor core's reads
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&m.conv[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (failed && lane == 0) {
            m.abort = 1;
            report(p.status, MOE_ERR_TIMEOUT);
        }
    } else if (kF4 && warp >= 6) {
        // ---------------- NVFP4 block-scale layout (warps 6..7) ----------------
        // A stage's block scales arrive row-major: row r's 16 bytes (the 16 blocks of
        // the stage's 256 elements) at 16 r, A rows then B rows, 2 KB each.  The MMA of
        // elements 64 kk .. 64 kk + 63 takes them as 512 bytes per operand: lane l's 16
        // bytes hold the 4 scales (blocks 4 kk .. 4 kk + 3) of rows l, 32 + l, 64 + l
        // and 96 + l.  Thread (l, pair) moves chunks 2 pair and 2 pair + 1 of both
        // operands: it reads all its words, the 64 threads meet, then write in place.
        const int ct = threadIdx.x - 6 * 32;  // 0 .. F4_CONV_THREADS - 1
        const int l = ct & 31, kp = (ct >> 5) * 2;
        uint32_t stage = 0, phase = 0;
        bool failed = false;
        if (ct == 0) m.conv_ok = mbar_wait(&m.ready, 0, p.timeout_ns, abortp) ? 1 : 0;
        asm volatile("bar.sync %0, %1;" ::"n"(CONV_BARRIER), "n"(F4_CONV_THREADS) : "memory");
        failed = !m.conv_ok;
        bool have = true;  // the prefix is published (waited for above)
        for (int iu = 0; !failed; ++iu) {
            const int u = next_unit(iu, have);
            if (u < 0) break;
            const Tile tl = tile_of<kFC1, kPair>(u, p, m, n_sh_tiles, mu_sh, crank);
            const int nkb = tl.kb1 - tl.kb0;
            for (int kb = 0; kb < nkb; ++kb) {
                if (ct == 0) m.conv_ok = mbar_wait(&m.full[stage], phase, p.timeout_ns, abortp) ? 1 : 0;
                asm volatile("bar.sync %0, %1;" ::"n"(CONV_BARRIER), "n"(F4_CONV_THREADS) : "memory");
                if (!m.conv_ok) {
                    failed = true;
                    break;
                }
                uint8_t* sfa = smSF + (size_t)stage * SF_STAGE_BYTES;
                const uint32_t* ra = reinterpret_cast<const uint32_t*>(sfa);
                const uint32_t* rb = reinterpret_cast<const uint32_t*>(sfa + SF_STAGE_BYTES / 2);
                uint32_t wa[2][4], wb[2][4];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        wa[c][q] = ra[(32 * q + l) * 4 + kp + c];
                        wb[c][q] = rb[(32 * q + l) * 4 + kp + c];
                    }
                asm volatile("bar.sync %0, %1;" ::"n"(CONV_BARRIER), "n"(F4_CONV_THREADS) : "memory");
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    *reinterpret_cast<uint4*>(sfa + (kp + c) * 512 + l * 16) =
                        make_uint4(wa[c][0], wa[c][1], wa[c][2], wa[c][3]);
                    *reinterpret_cast<uint4*>(sfa + SF_STAGE_BYTES / 2 + (kp + c) * 512 + l * 16) =
                        make_uint4(wb[c][0], wb[c][1], wb[c][2], wb[c][3]);
                }
                // generic-proxy stores -> visible to the tensor core's copies
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&m.conv[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (failed && lane == 0) {
            m.abort = 1;
            report(p.status, MOE_ERR_TIMEOUT);
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    if (kPair) {
        __syncwarp();        // lane 0 of warps 0 and 1 arrives late from its role loop
        cluster_sync_all();  // neither CTA leaves while its peer may still address it
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_ALLOC);
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

// bf16 (u8 = false) or byte (u8 = true) matrix [outer, inner]: boxes of one
// 128-byte row (64 bf16 or 128 bytes) x box_outer rows, 128-byte swizzle
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer,
               bool u8 = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t es_bytes = u8 ? 1 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * es_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(128 / es_bytes), box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 weights [groups, rows, inner] bytes: boxes of 64 bytes x box_rows rows, no
// swizzle (dense rows; the converter warps lay them out for the MMA)
bool encode_3d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t groups,
                  uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, groups};
    cuuint64_t strides[2] = {inner, rows * inner};
    cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 or byte matrices [groups, rows, inner]: boxes of one 128-byte row x
// box_rows rows of one group, 128-byte swizzle
bool encode_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t groups,
               uint32_t box_rows, bool u8 = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t es_bytes = u8 ? 1 : 2;
    cuuint64_t dims[3] = {inner, rows, groups};
    cuuint64_t strides[2] = {inner * es_bytes, rows * inner * es_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es_bytes), box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NVFP4 block scales [groups][rows][row_bytes] bytes (row_bytes a multiple of
// 16): boxes of 16 bytes (one pipeline stage's 16 blocks) x box_rows rows, no
// swizzle (the converter warps lay them out for the tensor core)
bool encode_sf(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t groups,
               uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {row_bytes, rows, groups};
    cuuint64_t strides[2] = {row_bytes, rows * row_bytes};
    cuuint32_t box[3] = {16, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device launch facts of one kernel instantiation: shared-memory limit set,
// and (pair mode) how many 2-CTA clusters can be resident at once.
struct KernelInfo {
    bool ready = false;
    int max_clusters = 0;
};

template <bool kFC1, bool kPair, int BN, bool kShort, int kQ>
cudaError_t kernel_info(int num_sms, KernelInfo* out) {
    static std::mutex mu;
    static KernelInfo info[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!info[dev].ready) {
        err = cudaFuncSetAttribute(grouped_gemm_kernel<kFC1, kPair, BN, kShort, kQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_bytes<kPair, BN, kShort, chunks_per_stage<kShort, kQ>(), sf_stage_bytes<kQ>()>());
        if (err != cudaSuccess) return err;
        int clusters = 0;
        if (kPair) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * num_sms);
            cfg.blockDim = dim3(threads_of<kQ>());
            cfg.dynamicSmemBytes = smem_bytes<kPair, BN, kShort, chunks_per_stage<kShort, kQ>(), sf_stage_bytes<kQ>()>();
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 2;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            err = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<kFC1, kPair, BN, kShort, kQ>, &cfg);
            if (err != cudaSuccess) return err;
        }
        info[dev].max_clusters = clusters;
        info[dev].ready = true;
    }
    *out = info[dev];
    return cudaSuccess;
}

template <bool kFC1, bool kPair, int BN, bool kShort, int kQ>
cudaError_t launch_kernel(const GemmParams& p, const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mAs,
                          const CUtensorMap& mBs, const CUtensorMap& mA32, const CUtensorMap& mAs32,
                          const CUtensorMap& mSFA, const CUtensorMap& mSFB, const CUtensorMap& mSFAs,
                          const CUtensorMap& mSFBs, unsigned grid,
                          cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads_of<kQ>());
    cfg.dynamicSmemBytes = smem_bytes<kPair, BN, kShort, chunks_per_stage<kShort, kQ>(), sf_stage_bytes<kQ>()>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (kPair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    char name[MOE_LAUNCH_LABEL_BYTES];
    snprintf(name, sizeof(name), "grouped_gemm_%s_n%d%s%s%s", kFC1 ? "fc1" : "fc2", BN, kShort ? "_short" : "",
             kPair ? "_pair" : "",
             kQ == GEMM_W8 ? "_w8" : (kQ == GEMM_W8A8 ? "_w8a8" : (kQ == GEMM_NVFP4 ? "_nvfp4" : "")));
    const cudaError_t e = note_launch(name, s);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<kFC1, kPair, BN, kShort, kQ>, p, mA, mB, mAs, mBs, mA32, mAs32,
                              mSFA, mSFB, mSFAs, mSFBs);
}

// Tensor maps, parameters and grid of one launch with MMA N = BN.
template <bool kFC1, bool kPair, int BN, bool kShort, int kQ>
cudaError_t launch_bn(const GemmLaunch& L, int num_sms, int64_t bound, cudaStream_t s, const char** why) {
    const bool has_routed = L.G > 0 && L.rows_cap > 0;
    const bool has_shared = L.T_sh > 0 && L.b_sh != nullptr && L.N_out_sh > 0;
    // B boxes: FC1 loads gate and up halves of BN/2 rows; FC2 BN rows (pair: 128)
    const uint32_t brows = kFC1 ? BN / 2 : (kPair ? BN / 2 : BN);
    CUtensorMap mA, mB, mAs, mBs, mA32, mAs32, mSFA, mSFB, mSFAs, mSFBs;
    bool ok = true;
    constexpr bool a8 = kQ == GEMM_W8A8;
    constexpr bool f4 = kQ == GEMM_NVFP4;
    // operand rows in bytes: K bf16 / E4M3 elements, or K / 2 bytes of packed E2M1
    const uint64_t ka = f4 ? (uint64_t)L.K / 2 : (uint64_t)L.K;
    const uint64_t ka_sh = f4 ? (uint64_t)L.K_sh / 2 : (uint64_t)L.K_sh;
    const bool u8 = a8 || f4;
    const uint32_t sfa_rows = kShort ? BM_SHORT : BM;
    if (has_routed) {
        ok = ok && encode_2d(&mA, L.a, ka, (uint64_t)L.rows_cap, BM, u8);
        ok = ok && encode_2d(&mA32, L.a, ka, (uint64_t)L.rows_cap, BM_SHORT, u8);
        ok = ok && (kQ == GEMM_W8 ? encode_3d_u8(&mB, L.b, (uint64_t)L.K, (uint64_t)L.Nb, (uint64_t)L.G, brows)
                                  : encode_3d(&mB, L.b, ka, (uint64_t)L.Nb, (uint64_t)L.G, brows, u8));
        if (f4) {
            ok = ok && encode_sf(&mSFA, L.a_sf, nvfp4_sf_row_bytes(L.K), (uint64_t)L.rows_cap, 1, sfa_rows);
            ok = ok && encode_sf(&mSFB, L.b_sf, nvfp4_sf_row_bytes(L.K), (uint64_t)L.Nb, (uint64_t)L.G, brows);
        }
    }
    if (has_shared) {
        ok = ok && encode_2d(&mAs, L.a_sh, ka_sh, (uint64_t)L.T_sh, BM, u8);
        ok = ok && encode_2d(&mAs32, L.a_sh, ka_sh, (uint64_t)L.T_sh, BM_SHORT, u8);
        ok = ok && (kQ == GEMM_W8 ? encode_3d_u8(&mBs, L.b_sh, (uint64_t)L.K_sh, (uint64_t)L.Nb_sh, 1, brows)
                                  : encode_3d(&mBs, L.b_sh, ka_sh, (uint64_t)L.Nb_sh, 1, brows, u8));
        if (f4) {
            ok = ok && encode_sf(&mSFAs, L.a_sf_sh, nvfp4_sf_row_bytes(L.K_sh), (uint64_t)L.T_sh, 1, sfa_rows);
            ok = ok && encode_sf(&mSFBs, L.b_sf_sh, nvfp4_sf_row_bytes(L.K_sh), (uint64_t)L.Nb_sh, 1, brows);
        }
    }
    if (!ok) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    if (!has_routed) {
        mA = mAs;
        mA32 = mAs32;
        mB = mBs;
        if (f4) {
            mSFA = mSFAs;
            mSFB = mSFBs;
        }
    }
    if (!has_shared) {
        mAs = mA;
        mAs32 = mA32;
        mBs = mB;
        if (f4) {
            mSFAs = mSFA;
            mSFBs = mSFB;
        }
    }
    if (!f4) {  // unused by the other formats
        mSFA = mSFB = mSFAs = mSFBs = mA;
    }
    GemmParams p;
    p.offsets = L.offsets;
    p.G = has_routed ? L.G : 0;
    p.K = L.K;
    p.K_sh = L.K_sh;
    p.N_out = L.N_out;
    p.N_out_sh = L.N_out_sh;
    p.up_off = kFC1 ? L.Nb / 2 : 0;
    p.up_off_sh = kFC1 ? L.Nb_sh / 2 : 0;
    p.rows_cap = L.rows_cap;
    p.T_sh = has_shared ? L.T_sh : 0;
    p.scale = L.b_scale;
    p.scale_sh = L.b_scale_sh;
    p.a_scale = L.a_scale;
    p.a_scale_sh = L.a_scale_sh;
    // K steps: 64 bf16 or 128 E4M3 elements (one 128-byte row); a ragged last step
    // of E4M3 operands is zero-filled by the TMA past K
    const int ke = f4 ? 4 * BK : (a8 ? 2 * BK : BK);
    p.kb_total = (L.K + ke - 1) / ke;
    p.kb_total_sh = (L.K_sh + ke - 1) / ke;
    p.Nb = L.Nb;
    p.out_sh_part = L.out_sh_part;
    p.ksplit_sh = (has_shared && !L.swiglu && L.out_sh_part && L.ksplit_sh > 1) ? L.ksplit_sh : 1;
    // ranges of a split shared tile hold whole stages (KSC chunks each)
    constexpr int KSC = chunks_per_stage<kShort, kQ>();
    p.kb_split_sh = (p.kb_total_sh + p.ksplit_sh - 1) / p.ksplit_sh;
    p.kb_split_sh = (p.kb_split_sh + KSC - 1) / KSC * KSC;
    // (measured: one token 6 % off the layer step, 8 and 32 tokens 1-2 %; at 128 tokens the
    // shared stream no longer fits in the window and the prefetch costs about 1 %)
    p.prefetch_sh = (kFC1 && has_shared && L.T_sh <= 64) ? 1 : 0;
    p.out = L.out;
    p.out_sh = L.out_sh;
    p.out_row = L.out_row;
    p.status = &L.hdr->status;
    p.timeout_ns = L.timeout_ns;

    KernelInfo info;
    cudaError_t err = kernel_info<kFC1, kPair, BN, kShort, kQ>(num_sms, &info);
    if (err != cudaSuccess) {
        *why = "kernel attribute / occupancy query failed";
        return err;
    }
    unsigned grid;
    if (kPair) {
        const int64_t units = (bound + 1) / 2;
        const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(units, std::max(1, info.max_clusters)));
        grid = (unsigned)(2 * clusters);
    } else {
        grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(bound, num_sms));
    }
    err = launch_kernel<kFC1, kPair, BN, kShort, kQ>(p, mA, mB, mAs, mBs, mA32, mAs32, mSFA, mSFB, mSFAs, mSFBs, grid,
                                                    s);
    if (err != cudaSuccess) *why = "launch failed";
    return err;
}

// Upper bound of the tiles of a launch with MMA N = bn (single CTAs): at most
// min(G, rows) groups are non-empty, each adding at most one partial m-tile.
// K ranges of the shared problem: FC2 only, when the caller supplied a partial buffer
int split_of(const GemmLaunch& L) {
    return (!L.swiglu && L.out_sh_part && L.ksplit_sh > 1) ? L.ksplit_sh : 1;
}

int64_t tile_bound(const GemmLaunch& L, int bn) {
    const int ow = L.swiglu ? bn / 2 : bn;
    int64_t bound = 0;
    if (L.G > 0 && L.rows_cap > 0)
        bound += (int64_t)((L.N_out + ow - 1) / ow) *
                 ((L.rows_cap + BM - 1) / BM + std::min<int64_t>(L.G, L.rows_cap));
    if (L.T_sh > 0 && L.b_sh != nullptr && L.N_out_sh > 0)
        bound += (int64_t)((L.N_out_sh + ow - 1) / ow) * ((L.T_sh + BM - 1) / BM) * split_of(L);
    return bound;
}

template <bool kFC1>
cudaError_t dispatch(const GemmLaunch& L, int num_sms, cudaStream_t s, const char** why) {
    const int64_t b256 = tile_bound(L, 256);
    if (L.quant == GEMM_W8) {
        // E4M3 weights: N = 256, single CTAs; 32-row A slots when every tile is short
        if (L.max_group_rows <= BM_SHORT && L.T_sh <= BM_SHORT)
            return launch_bn<kFC1, false, 256, true, GEMM_W8>(L, num_sms, b256, s, why);
        return launch_bn<kFC1, false, 256, false, GEMM_W8>(L, num_sms, b256, s, why);
    }
    if (L.quant == GEMM_NVFP4) {
        // E2M1 operands with block scales: single CTAs, N = 128 (the accumulators and
        // the scales' tensor-memory columns fit one allocation)
        const int64_t b128 = tile_bound(L, 128);
        if (L.max_group_rows <= BM_SHORT && L.T_sh <= BM_SHORT)
            return launch_bn<kFC1, false, 128, true, GEMM_NVFP4>(L, num_sms, b128, s, why);
        return launch_bn<kFC1, false, 128, false, GEMM_NVFP4>(L, num_sms, b128, s, why);
    }
    if (L.quant == GEMM_W8A8) {
        // E4M3 operands: single CTAs, tile widths chosen as for bf16
        if (L.max_group_rows <= BM_SHORT && L.T_sh <= BM_SHORT)
            return launch_bn<kFC1, false, 256, true, GEMM_W8A8>(L, num_sms, b256, s, why);
        if (L.rows_cap <= 1024 || b256 >= 2 * (int64_t)num_sms)
            return launch_bn<kFC1, false, 256, false, GEMM_W8A8>(L, num_sms, b256, s, why);
        const int64_t b128 = tile_bound(L, 128);
        if (b128 >= 2 * (int64_t)num_sms)
            return launch_bn<kFC1, false, 128, false, GEMM_W8A8>(L, num_sms, b128, s, why);
        return launch_bn<kFC1, false, 64, false, GEMM_W8A8>(L, num_sms, tile_bound(L, 64), s, why);
    }
    const bool pair = split_of(L) == 1 &&
                      (L.pair_mode == 2 ? b256 >= 2 : (L.pair_mode == 1 && b256 >= 4 * (int64_t)num_sms));
    if (pair) return launch_bn<kFC1, true, 256, false, GEMM_BF16>(L, num_sms, b256, s, why);
    // every tile at most 32 rows: 32-row A slots, so more stages fit the ring
    if (L.max_group_rows <= BM_SHORT && L.T_sh <= BM_SHORT)
        return launch_bn<kFC1, false, 256, true, GEMM_BF16>(L, num_sms, b256, s, why);
    // Small batches (at most 1024 routed rows) stream weights: N = 256 moves the
    // most bytes per pipeline stage, and a stage costs about the same time
    // whatever its size, so the widest tile wins even with SMs left idle.
    // Otherwise the widest N that still gives every SM two tiles.
    if (L.rows_cap <= 1024 || b256 >= 2 * (int64_t)num_sms)
        return launch_bn<kFC1, false, 256, false, GEMM_BF16>(L, num_sms, b256, s, why);
    const int64_t b128 = tile_bound(L, 128);
    if (b128 >= 2 * (int64_t)num_sms) return launch_bn<kFC1, false, 128, false, GEMM_BF16>(L, num_sms, b128, s, why);
    return launch_bn<kFC1, false, 64, false, GEMM_BF16>(L, num_sms, tile_bound(L, 64), s, why);
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
    return L.swiglu ? dispatch<true>(L, num_sms, s, why) : dispatch<false>(L, num_sms, s, why);
}

cudaError_t launch_wait_timeout_probe(WsHeader* hdr, uint64_t timeout_ns, cudaStream_t s) {
    const cudaError_t e = note_launch("wait_probe", s);
    if (e != cudaSuccess) return e;
    wait_probe_kernel<<<1, 32, 0, s>>>(&hdr->status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace moe
