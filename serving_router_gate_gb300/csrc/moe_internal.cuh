// moe_internal.cuh -- device helpers shared by the kernels of the GB300 MoE
// layer: status word, bounded waits, mbarrier / TMA / tcgen05 inline PTX.
// Internal to the library (not installed); the public ABI is include/moe.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Workspace header (first kWsHeaderBytes bytes of every workspace)
// ---------------------------------------------------------------------------
constexpr size_t kWsHeaderBytes = MOE_WS_HEADER_BYTES;
struct WsHeader {
    int32_t status;              // OR of MOE_ERR_DEVICE_BOUNDS / MOE_ERR_TIMEOUT
    int32_t pad0;
    unsigned long long refined;  // tokens whose top-k needed the fp64 recheck
    unsigned int route_ticket;   // small-batch router: CTAs of the running launch that have
                                 // written their logits (back to 0 when the launch ends)
};

__device__ __forceinline__ void report(int32_t* status, int32_t code) {
    if (status) atomicOr(status, code);
}

// Bounds check of a global index that data (offsets, ranks, ids) decides.  The
// library built with MOE_CHECKED tests 0 <= i < n, reports MOE_ERR_DEVICE_BOUNDS
// and skips the access when it fails; the regular build assumes it (every such
// index is derived from values the kernels validate where they are read).
#ifdef MOE_CHECKED
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n, int32_t* status) {
    if (i >= 0 && i < n) return true;
    report(status, MOE_ERR_DEVICE_BOUNDS);
    return false;
}
#else
__device__ __forceinline__ bool in_bounds(int64_t, int64_t, int32_t*) { return true; }
#endif

// ---------------------------------------------------------------------------
// bf16 helpers (bit patterns in uint16_t)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// Time and bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream finishes;
// it must wait (pdl_wait) before touching memory that kernel writes or reads.
// pdl_trigger lets the next kernel on the stream be scheduled early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed.  Gives up
// (returns false) once `timeout_ns` has passed since the wait began, or as soon
// as *abort becomes nonzero; never spins without a bound.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* abort) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t polls = 0;
    while (true) {
        if (mbar_try_wait(a, parity)) return true;
        if ((++polls & 255u) == 0u) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor): every load lands in the issuing CTA (or, for the
// cta_group::2 forms below, in its own half of a pair); no load is multicast
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Pull `bytes` (a multiple of 16, from a 16-byte-aligned address) of global memory
// into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// Pull one box of a tensor into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives and waits (release/acquire).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in the CTA of rank `rank` of this
// cluster (a shared::cluster address).
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in a peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA loads for 2-CTA (cta_group::2) MMAs: the box lands in this CTA's shared
// memory and the completed bytes are signalled on the mbarrier at
// `bar_cluster` (a shared::cluster address, here the pair leader's barrier).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
        : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= (A x SFA)[smem] * (B x SFB)[smem]^T, packed E2M1 inputs with one
// E4M3 scale per 16 elements (kind::mxf4nvf4, scale_vec::4X; K = 64 per
// instruction: 32 bytes of a 128-byte row), fp32 accumulation.  The scales of
// the instruction's 4 K blocks sit in 4 tensor-memory columns from sfa / sfb:
// row r's four scale bytes (K-block order) in lane r % 32 of every lane
// quarter, column r / 32.
__device__ __forceinline__ void tc_mma_nvfp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy 32 rows x 16 bytes of shared memory (rows contiguous, from a 16-byte
// aligned address) into 4 tensor-memory columns from `taddr`, row i to lane i of
// every lane quarter.
__device__ __forceinline__ void tc_copy_32x128b_x4(uint32_t taddr, uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 32;  // 8-row core matrices of 16-byte rows, 128 bytes apart
    d |= (uint64_t)1 << 46;           // descriptor version
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 inputs (kind::f8f6f4, K = 32 per
// instruction: 32 bytes of a 128-byte row, as for bf16), fp32 accumulation.
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// As tc_commit, arriving on the mbarrier at `bar`'s offset in every CTA of the
// cluster named in cta_mask.
__device__ __forceinline__ void tc_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ---- 2-CTA (cta_group::2) forms: one MMA spans the two CTAs of a cluster pair.
// A's rows and B's rows are split between the CTAs (rank 0: first half), both at
// the same shared-memory offsets; each CTA's TMEM receives its half of D's rows.
// Allocation, relinquish and deallocation are executed by one warp in each CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the mbarrier at `bar`'s offset in the CTAs of cta_mask when this
// thread's prior 2-CTA tcgen05 operations complete
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 64 elements (128 B), 8-row groups 1024 B apart.
// The tile base must be 1024-byte aligned; stepping K by 16 elements inside the
// 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address (16-byte units)
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                        // descriptor version
    d |= (uint64_t)2 << 61;                        // swizzle: 128 B
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 A and B (both
// K-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                              // D format: f32
           | (1u << 7)                            // A format: bf16
           | (1u << 10)                           // B format: bf16
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Instruction descriptor of tcgen05.mma.kind::mxf4nvf4: E2M1 A and B (format
// code 1, K-major), E4M3 block scales (scale format 0), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int M, int N) {
    return (1u << 7)                              // A format: E2M1
           | (1u << 10)                           // B format: E2M1
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4: E4M3 A and B (format
// code 0 in both fields, both K-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                              // D format: f32
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// ---------------------------------------------------------------------------
// Internal launchers (defined in the kernel files, called by moe_api.cu)
// ---------------------------------------------------------------------------
struct RouterLaunch {
    const uint16_t* x;
    const float* Wg;
    const float* bias;
    int64_t T;
    int H, E, k, renorm;
    int32_t* ids;
    float* w;
    float* part;   // [nsplit][T][E]
    float* xsq;    // [nsplit][T]
    float* wsq;    // [nsplit][E]
    int nsplit, KC;
    int n_group = 1, topk_group = 1;  // group-limited top-k (n_group <= 1: every expert eligible)
    WsHeader* hdr;
};
size_t router_scratch_bytes(int64_t T, int H, int E, int num_sms);
void router_carve(void* base, int64_t T, int E, float** part, float** xsq, float** wsq);
void router_plan(int64_t T, int H, int E, int num_sms, int* nsplit, int* KC);
cudaError_t launch_router(const RouterLaunch& L, int num_sms, cudaStream_t s);

struct PermuteLaunch {
    const int32_t* ids;
    float* w;
    int64_t T;
    int k, E;
    const int32_t* rep_offset;
    const int32_t* rep_slots;
    int S, local_start, local_count, mode, S_local;
    const uint16_t* x;
    int H;
    int32_t* slot_ids;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm_src;
    int32_t* pair_row;
    uint16_t* x_perm;
    int32_t* rank;        // [T*k] rank of each pair among its chunk's pairs of its slot
    int32_t* chunk_cnt;   // [nchunks][S_local]
    int32_t* chunk_base;  // [nchunks][S_local]
    bool scale_rows;      // x_perm rows = bf16(w * x) (routing applied on the input)
    WsHeader* hdr;
};
size_t permute_scratch_bytes(int64_t P, int S_local);
void permute_carve(void* base, int64_t P, int S_local, int32_t** rank, int32_t** chunk_cnt, int32_t** chunk_base);
cudaError_t launch_permute(const PermuteLaunch& L, int num_sms, cudaStream_t s);

struct GemmLaunch {
    bool swiglu;               // FC1 (gate/up pairs, SwiGLU epilogue) or FC2
    const uint16_t* a;         // routed A [rows_cap, K]
    int64_t rows_cap;
    const int32_t* offsets;    // [G+1]
    int G;
    const uint16_t* b;         // routed B [G, Nb, K]
    int K, Nb, N_out;          // Nb rows of B per group; N_out output columns
    uint16_t* out;             // [rows_cap, N_out]
    const int32_t* out_row = nullptr;  // or [rows_cap]: routed row r is stored at out row out_row[r]
    const uint16_t* a_sh;      // shared A [T_sh, K_sh] (or null)
    int64_t T_sh;
    const uint16_t* b_sh;      // shared B [Nb_sh, K_sh]
    int K_sh, Nb_sh, N_out_sh;
    uint16_t* out_sh;          // [T_sh, N_out_sh]
    float* out_sh_part;        // FC2 only, or null: split the shared problem's K into ksplit_sh ranges
    int ksplit_sh;             // and write fp32 partials [ksplit_sh, T_sh, N_out_sh] here (out_sh unused)
    WsHeader* hdr;
    uint64_t timeout_ns;
    int pair_mode;             // 0 single CTAs only, 1 pairs for large launches, 2 pairs whenever possible
    int64_t max_group_rows;    // upper bound on the rows of any routed group (tokens of the batch)
    int quant;                 // GEMM_BF16, GEMM_W8 (E4M3 B, bf16 A) or GEMM_W8A8 (E4M3 A and B)
    const float* b_scale;      // [G][Nb] row scales of b (E4M3 B only)
    const float* b_scale_sh;   // [Nb_sh] row scales of b_sh (E4M3 B only)
    const float* a_scale;      // [rows_cap] row scales of a (GEMM_W8A8 only)
    const float* a_scale_sh;   // [T_sh] row scales of a_sh (GEMM_W8A8 only)
    // GEMM_NVFP4: a, b, a_sh, b_sh hold packed E2M1 codes ([rows][K/2] bytes), these
    // their E4M3 block scales ([rows][nvfp4_sf_row_bytes(K)] bytes); b_scale / a_scale
    // hold the fp32 row scales
    const uint8_t* a_sf = nullptr;
    const uint8_t* a_sf_sh = nullptr;
    const uint8_t* b_sf = nullptr;
    const uint8_t* b_sf_sh = nullptr;
};
enum { GEMM_BF16 = 0, GEMM_W8 = 1, GEMM_W8A8 = 2, GEMM_NVFP4 = 3 };
cudaError_t launch_grouped_gemm(const GemmLaunch& L, int num_sms, cudaStream_t s, const char** why);

struct FinalizeLaunch {
    const uint16_t* y;
    int64_t rows_cap;
    const int32_t* pair_row;
    const float* w;
    int64_t T;
    int k, H;
    const uint16_t* y_sh;
    const float* y_sh_part;    // or null: fp32 partials [ksplit, T, H] of the shared expert, summed in order
    int ksplit;
    const uint16_t* x;
    const uint16_t* gate_w;
    uint16_t* out;
    WsHeader* hdr;
};
cudaError_t launch_finalize(const FinalizeLaunch& L, int num_sms, cudaStream_t s);

// Rows of an all-to-all expert-parallel rank between exchange order and GEMM order
// (moe_a2a_regroup).
struct A2aRegroupLaunch {
    const int32_t* recv_counts;  // [N, S_local]
    int N, S_local;
    int64_t rows_cap;
    int H;
    const uint16_t* src;
    uint16_t* dst;
    bool to_exchange;            // false: exchange -> GEMM order; true: GEMM -> exchange order
    int32_t* offsets;            // [S_local + 1] GEMM-order slot offsets, or null
    int32_t* row_map;            // [rows_cap]: for each destination row, its source row; or null
    WsHeader* hdr;
};
constexpr int kA2aMaxBlocks = 4096;  // N * S_local the shared-memory tables hold
size_t a2a_regroup_smem_bytes(int N, int S_local);
cudaError_t launch_a2a_regroup(const A2aRegroupLaunch& L, int num_sms, cudaStream_t s);

// The one reduction of expert parallelism by plain loads of the ranks' partials
// (moe_ep_signal, moe_ep_reduce).
constexpr int kEpMaxRanks = 16;
struct EpReduceLaunch {
    const uint16_t* partials[kEpMaxRanks];  // [T, H] bf16 partial of each rank (peer-mapped pointers)
    int N;
    const int32_t* flags;                    // [N] this rank's flags
    int32_t epoch;
    int64_t row0, row1;
    int H;
    uint16_t* out;
    uint64_t timeout_ns;
    WsHeader* hdr;
};
cudaError_t launch_ep_signal(int32_t* const* peer_flags, int N, int rank, int32_t epoch, cudaStream_t s);
cudaError_t launch_ep_reduce(const EpReduceLaunch& L, int num_sms, cudaStream_t s);

cudaError_t launch_wait_timeout_probe(WsHeader* hdr, uint64_t timeout_ns, cudaStream_t s);

// Row-wise E4M3 quantisation of a bf16 matrix [rows, K] (moe_quantize_fp8_rows).
// E4M3 activation rows with power-of-two scales: up to two row sets per launch;
// a set with rows_dev takes min(rows, *rows_dev) rows, read on the device.
struct ActQuantSeg {
    const uint16_t* src;       // [rows, K] bf16
    int64_t rows;
    const int32_t* rows_dev;   // or null
    int K;
    uint8_t* dst;              // [rows, K], or null
    float* scale;              // [rows]
    // optional: row t's codes and scale also go to rows pair_row[t * k + j] (j < k;
    // -1 and rows past dst2_rows skipped) of dst2 / scale2
    const int32_t* pair_row;
    int k;
    uint8_t* dst2;
    float* scale2;
    int64_t dst2_rows;
};
cudaError_t launch_quantize_act_rows(const ActQuantSeg* seg, int nseg, int num_sms, cudaStream_t s);
cudaError_t launch_quantize_fp8_rows(const uint16_t* w, int64_t rows, int K, uint8_t* q, float* scale, int num_sms,
                                     cudaStream_t s);

// NVFP4 quantisation of bf16 rows [rows, K] (K a multiple of 64): packed E2M1
// codes [rows][K/2], E4M3 block scales [rows][16 * ceil(K / 256)] (zero past
// K / 16) and fp32 row scales [rows]; pow2: power-of-two row scales
// (activations), else amax / 2688 (weights).  A segment with rows_dev takes
// min(rows, *rows_dev) rows, read on the device.
struct Nvfp4QuantSeg {
    const uint16_t* src;       // [rows, K] bf16
    int64_t rows;
    const int32_t* rows_dev;   // or null
    int K;
    int pow2;
    uint8_t* q;                // [rows, K/2] codes, or null
    uint8_t* sb;               // [rows, nvfp4_sf_row_bytes(K)] block scales
    float* scale;              // [rows] row scales
    // optional: row t's codes and scales also go to rows pair_row[t * k + j] (j < k;
    // -1 and rows past dst2_rows skipped) of q2 / sb2 / scale2
    const int32_t* pair_row = nullptr;
    int k = 0;
    uint8_t* q2 = nullptr;
    uint8_t* sb2 = nullptr;
    float* scale2 = nullptr;
    int64_t dst2_rows = 0;
};
cudaError_t launch_quantize_nvfp4_rows(const Nvfp4QuantSeg* seg, int nseg, int num_sms, cudaStream_t s);
// bytes of one row of NVFP4 block scales
__host__ __device__ constexpr int nvfp4_sf_row_bytes(int K) { return 16 * ((K + 255) / 256); }

// Whether kernels are launched with programmatic stream serialization (set by
// moe_set_pdl; defined in moe_api.cu).
bool pdl_enabled();
// Called right before each kernel launch: adds one to the library's count of
// launches (moe_get_launch_count) and, while the launch-event hook is armed,
// records its next event on `s` labelled `name` (moe_launch_events_arm).  A
// non-success return means the launch must not be made.
cudaError_t note_launch(const char* name, cudaStream_t s);

// Launch `kernel` on `s`, with programmatic stream serialization when enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    const cudaError_t e = note_launch(name, s);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
