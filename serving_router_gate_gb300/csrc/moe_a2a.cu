// moe_a2a.cu -- the row reorder of one rank of the all-to-all expert-parallel
// layer.
//
// Method: TensorRT-LLM PR #10985, "MoE all-to-all paradigm", sequence diagram
// (all-to-all path): the fused op dispatches the tokens to the ranks
// responsible for their experts, each rank computes the MoE on its local
// experts, and the results are gathered back to the tokens' ranks.
//
// A rank sends its permuted rows (moe_permute groups them by slot, and the slots
// of one destination rank are a contiguous range), so what a rank receives is in
// EXCHANGE order: source rank 0's rows, then rank 1's, ...; inside one source's
// block, its rows of local slot 0, then slot 1, ...  The grouped GEMMs want GEMM
// order: slot 0's rows, then slot 1's, ...; inside one slot, the rows of source
// 0, then source 1, ... (each source's rows keep their order).  Block (n, c) =
// the cnt[n][c] rows source n sent for local slot c:
//   exchange start  X(n, c) = sum of cnt over the blocks before (n, c) in (n, c) order,
//   GEMM start      G(n, c) = sum of cnt over the blocks before (n, c) in (c, n) order,
// and row q = X(n, c) + i of the exchange order is row G(n, c) + i of the GEMM
// order (0 <= i < cnt[n][c]).  The GEMM-order slot offsets are G(0, c).
//
// One kernel moves rows either way (a pure copy; HBM-bound: 2 x rows x H x 2
// bytes) and can record, for each destination row, its source row (with the
// GEMM order as destination, that map lets FC2 store its output rows straight
// back in exchange order).  Each CTA loads the N x S_local counts into shared
// memory, forms X and G with two block-wide scans, and its warps then take rows
// of the exchange order grid-stride: a binary search over X finds the row's
// block, and the warp's lanes copy the row as 16-byte vectors, several loads in
// flight per lane before the stores.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int A2A_THREADS = 256;
constexpr int A2A_WARPS = A2A_THREADS / 32;
constexpr int A2A_UNROLL = 4;  // 16-byte vectors a lane loads before it stores

// Exclusive prefix sums over nb entries in an order given by pos -> entry index:
// out[idx(p)] = sum_{p' < p} val[idx(p')].  val and out may be the same array
// (each thread reads an entry before it writes it, and its entries are its own).
// Returns the total.  Called by every thread of the CTA.
template <typename Idx>
__device__ int64_t block_exclusive_scan(const int32_t* val, int32_t* out, int nb, Idx idx, int64_t* warp_sum) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int per = (nb + A2A_THREADS - 1) / A2A_THREADS;
    const int p0 = min(nb, t * per), p1 = min(nb, p0 + per);
    int64_t local = 0;
    for (int p = p0; p < p1; ++p) local += val[idx(p)];
    int64_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    int64_t base = 0, total = 0;
    for (int i = 0; i < A2A_WARPS; ++i) {
        const int64_t s = warp_sum[i];
        if (i < w) base += s;
        total += s;
    }
    int64_t run = base + incl - local;
    for (int p = p0; p < p1; ++p) {
        const int e = idx(p);
        const int32_t v = val[e];
        out[e] = (int32_t)run;
        run += v;
    }
    __syncthreads();  // warp_sum is reused by the next scan
    return total;
}

__global__ void __launch_bounds__(A2A_THREADS, 4)
a2a_regroup_kernel(const int32_t* __restrict__ cnt_g, int N, int S_l, int64_t rows_cap,
                   const uint4* __restrict__ src, uint4* __restrict__ dst, int row_vecs, int to_exchange,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ row_map, int32_t* status) {
    extern __shared__ int32_t a2a_sm[];
    int32_t* X = a2a_sm;                // [N * S_l] exchange-order starts, then (first) the counts
    int32_t* G = a2a_sm + N * S_l;      // [N * S_l] GEMM-order starts
    __shared__ int64_t warp_sum[A2A_WARPS];
    __shared__ int bad;
    const int nb = N * S_l;

    pdl_wait();  // the counts and the source rows come from the previous work on the stream
    pdl_trigger();
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += A2A_THREADS) {
        const int32_t v = cnt_g[b];
        if (v < 0) bad = 1;
        X[b] = v;
    }
    __syncthreads();
    // GEMM order first (it reads the counts held in X), then the exchange order in place
    block_exclusive_scan(X, G, nb, [=](int p) { return (p % N) * S_l + p / N; }, warp_sum);
    const int64_t total = block_exclusive_scan(X, X, nb, [](int p) { return p; }, warp_sum);
    if (bad || total > rows_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(status, MOE_ERR_DEVICE_BOUNDS);
        return;
    }
    if (offsets && blockIdx.x == 0) {
        for (int c = threadIdx.x; c < S_l; c += A2A_THREADS) offsets[c] = G[c];  // block (0, c)
        if (threadIdx.x == 0) offsets[S_l] = (int32_t)total;
    }

    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * A2A_WARPS;
    for (int64_t q = (int64_t)blockIdx.x * A2A_WARPS + (threadIdx.x >> 5); q < total; q += nwarps) {
        // the row's block: the last b with X[b] <= q (an empty block shares its start
        // with the next one, so the search never ends on an empty block)
        int lo = 0, hi = nb;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (X[mid] <= q) lo = mid + 1;
            else hi = mid;
        }
        const int b = lo - 1;
        const int64_t r = (int64_t)G[b] + (q - X[b]);
        const int64_t from = to_exchange ? r : q, to = to_exchange ? q : r;
        if (!in_bounds(from, rows_cap, status) || !in_bounds(to, rows_cap, status)) continue;
        if (row_map && lane == 0) row_map[to] = (int32_t)from;
        const uint4* s = src + from * row_vecs;
        uint4* d = dst + to * row_vecs;
        for (int v0 = lane; v0 < row_vecs; v0 += 32 * A2A_UNROLL) {
            uint4 buf[A2A_UNROLL];
#pragma unroll
            for (int u = 0; u < A2A_UNROLL; ++u)
                if (v0 + 32 * u < row_vecs) buf[u] = __ldg(s + v0 + 32 * u);
#pragma unroll
            for (int u = 0; u < A2A_UNROLL; ++u)
                if (v0 + 32 * u < row_vecs) d[v0 + 32 * u] = buf[u];
        }
    }
}

}  // namespace

size_t a2a_regroup_smem_bytes(int N, int S_local) { return (size_t)2 * N * S_local * sizeof(int32_t); }

cudaError_t launch_a2a_regroup(const A2aRegroupLaunch& L, int num_sms, cudaStream_t s) {
    const size_t smem = a2a_regroup_smem_bytes(L.N, L.S_local);
    // one warp per row at least; at most four CTAs per SM (grid-stride beyond)
    const int64_t want = (L.rows_cap + A2A_WARPS - 1) / A2A_WARPS;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 4));
    return launch_k("a2a_regroup_kernel", a2a_regroup_kernel, dim3(grid), dim3(A2A_THREADS), smem, s, L.recv_counts,
                    L.N, L.S_local, L.rows_cap, reinterpret_cast<const uint4*>(L.src), reinterpret_cast<uint4*>(L.dst),
                    L.H / 8, L.to_exchange ? 1 : 0, L.offsets, L.row_map, &L.hdr->status);
}

}  // namespace moe
