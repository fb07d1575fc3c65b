// moe_ep_reduce.cu -- the one reduction of expert parallelism, as plain loads of
// the ranks' partial outputs.
//
// Method: vLLM EP FusedMoE patch, ep_reduce_output (each rank's routed plus
// shared partial output, then one SUM over the ranks) and
// ep_reduce_scatter_output (the same sum, each rank keeping a slice of the
// rows); DeepSpeed PR #6964 (one reduction per layer, after the weighted sum
// of the selected experts' outputs).
//
// Each rank writes its bf16 partial [T, H] into a buffer every rank can read
// (its own GPU's memory, mapped into the peers' address spaces), then
// ep_signal_kernel raises the rank's flag in every rank's flag array to the
// step's epoch (a system-scope release after a system-scope fence, so the
// partial is visible before the flag).  ep_reduce_kernel waits until every
// rank's flag has reached the epoch -- one thread polls with system-scope
// acquire loads, for at most the library's wait limit, and on timeout flags
// MOE_ERR_TIMEOUT and writes nothing -- then sums, for its rows, the N partial
// rows in rank order in fp32 and rounds once to bf16.  16-byte vectors, grid
// stride; each thread issues its N loads before it sums them.  Traffic: N x rows
// x H x 2 bytes read (N - 1 of them from peers), rows x H x 2 written.
//
// Flags only grow (a rank's flag holds the last epoch it signalled), so a
// reader waits for flag - epoch >= 0, and a peer one step ahead does not stall
// it.  The partial buffers alternate by epoch parity: a rank writes slot
// e % 2 at step e only after its reduce of step e - 1 saw every rank's step
// e - 1 flag, and each rank raises that flag only after its own reduce of step
// e - 2 -- the last reader of slot e % 2 -- has completed on its stream.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int EPR_THREADS = 256;

struct EpPtrs {
    const uint4* p[kEpMaxRanks];
};
struct EpFlagPtrs {
    int32_t* p[kEpMaxRanks];
};

__device__ __forceinline__ int32_t ld_acquire_sys(const int32_t* a) {
    int32_t v;
    asm volatile("ld.acquire.sys.global.s32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_sys(int32_t* a, int32_t v) {
    asm volatile("st.release.sys.global.s32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

__global__ void ep_signal_kernel(EpFlagPtrs f, int N, int rank, int32_t epoch) {
    pdl_wait();  // the partial is written by the previous kernel on the stream
    if (threadIdx.x == 0) {
        __threadfence_system();
        for (int n = 0; n < N; ++n) st_release_sys(f.p[n] + rank, epoch);
    }
}

// MAXN: the largest rank count of the instantiation (the loads in flight per thread)
template <int MAXN>
__global__ void __launch_bounds__(EPR_THREADS)
ep_reduce_kernel(EpPtrs P, int N, const int32_t* __restrict__ flags, int32_t epoch, int64_t row0, int64_t row1,
                 int row_vecs, uint4* __restrict__ out, uint64_t timeout_ns, int32_t* status) {
    __shared__ int ok;
    pdl_wait();
    if (threadIdx.x == 0) {
        // every rank's flag at this epoch or later (wrap-safe), within the time limit
        bool all = true;
        const uint64_t t0 = globaltimer_ns();
        for (int n = 0; n < N && all; ++n) {
            while ((int32_t)(ld_acquire_sys(flags + n) - epoch) < 0) {
                if (globaltimer_ns() - t0 > timeout_ns) {
                    all = false;
                    break;
                }
                __nanosleep(256);
            }
        }
        ok = all ? 1 : 0;
        if (!all && blockIdx.x == 0) report(status, MOE_ERR_TIMEOUT);
    }
    __syncthreads();
    if (!ok) return;
    pdl_trigger();
    const int64_t nvec = (row1 - row0) * row_vecs;
    const int64_t base = row0 * row_vecs;
    const int64_t stride = (int64_t)gridDim.x * EPR_THREADS;
    for (int64_t i = (int64_t)blockIdx.x * EPR_THREADS + threadIdx.x; i < nvec; i += stride) {
        uint4 v[MAXN];
#pragma unroll
        for (int n = 0; n < MAXN; ++n)
            if (n < N) v[n] = __ldcg(P.p[n] + base + i);  // L2 (coherent) path: written by other GPUs
        float acc[8];
        unpack8(v[0], acc);  // rank 0's values exactly, then ranks 1 .. N-1 added in order
#pragma unroll
        for (int n = 1; n < MAXN; ++n) {
            if (n < N) {
                float f[8];
                unpack8(v[n], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] += f[e];
            }
        }
        out[base + i] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
}

}  // namespace

cudaError_t launch_ep_signal(int32_t* const* peer_flags, int N, int rank, int32_t epoch, cudaStream_t s) {
    EpFlagPtrs f = {};
    for (int n = 0; n < N; ++n) f.p[n] = peer_flags[n];
    return launch_k("ep_signal_kernel", ep_signal_kernel, dim3(1), dim3(32), 0, s, f, N, rank, epoch);
}

cudaError_t launch_ep_reduce(const EpReduceLaunch& L, int num_sms, cudaStream_t s) {
    EpPtrs P = {};
    for (int n = 0; n < L.N; ++n) P.p[n] = reinterpret_cast<const uint4*>(L.partials[n]);
    const int row_vecs = L.H / 8;
    const int64_t nvec = (L.row1 - L.row0) * row_vecs;
    const int64_t want = (nvec + EPR_THREADS - 1) / EPR_THREADS;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    auto go = [&](auto kernel) {
        return launch_k("ep_reduce_kernel", kernel, dim3(grid), dim3(EPR_THREADS), 0, s, P, L.N, L.flags, L.epoch,
                        L.row0, L.row1, row_vecs, reinterpret_cast<uint4*>(L.out), L.timeout_ns, &L.hdr->status);
    };
    if (L.N <= 2) return go(ep_reduce_kernel<2>);
    if (L.N <= 4) return go(ep_reduce_kernel<4>);
    if (L.N <= 8) return go(ep_reduce_kernel<8>);
    return go(ep_reduce_kernel<kEpMaxRanks>);
}

}  // namespace moe
