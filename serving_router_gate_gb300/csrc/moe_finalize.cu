// moe_finalize.cu -- unpermute and routing-weighted combine of each token's
// k expert outputs, plus the (optionally sigmoid-gated) shared expert.
//
// Method: DeepSpeed PR #6964 (AutoTP for MoE models): the layer output is the
// weighted sum of the outputs of the selected experts, formed once per layer;
// vLLM EP FusedMoE patch, ep_reduce_output: the shared expert's output is added
// to the routed output (out = routed_out + shared_out).  The shared gate
// sigmoid(x . w_s) is the Qwen2-MoE-style scaled shared expert.
//
// One CTA per token (grid-stride).  Each thread owns 8 consecutive columns
// (one 16-byte vector) at a time and accumulates in fp32 in fixed j order:
//   acc = fma(w_j, y[row_j], acc) for j = 0..k-1 (rows of -1 skipped),
//   acc = fma(g, y_shared, acc), out = bf16_rn(acc).
// The gate dot product x . w_s is reduced in a fixed order (per-thread strided
// partials, warp xor-butterfly, warps in index order), so results are
// bit-reproducible.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int FZ_THREADS = 256;
constexpr int FZ_MAXK = 32;

__global__ void __launch_bounds__(FZ_THREADS) finalize_kernel(
    const uint16_t* __restrict__ y, int64_t rows_cap, const int32_t* __restrict__ pair_row,
    const float* __restrict__ w, int64_t T, int k, int H, const uint16_t* __restrict__ y_sh,
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gate_w, uint16_t* __restrict__ out,
    int32_t* status) {
    __shared__ int64_t s_row[FZ_MAXK];
    __shared__ float s_w[FZ_MAXK];
    __shared__ float s_red[FZ_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vec = H / 8;

    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        if (tid < k) {
            const int32_t r = pair_row[t * k + tid];
            int64_t rr = r;
            if (r < -1 || r >= rows_cap) {
                report(status, MOE_ERR_DEVICE_BOUNDS);
                rr = -1;
            }
            s_row[tid] = rr;
            s_w[tid] = w[t * k + tid];
        }
        float g = 1.0f;
        if (y_sh && gate_w) {
            const uint4* xv = reinterpret_cast<const uint4*>(x + t * H);
            const uint4* gv = reinterpret_cast<const uint4*>(gate_w);
            float d = 0.f;
            for (int v = tid; v < vec; v += FZ_THREADS) {
                float a[8], b[8];
                unpack8(__ldg(xv + v), a);
                unpack8(__ldg(gv + v), b);
#pragma unroll
                for (int i = 0; i < 8; ++i) d = fmaf(a[i], b[i], d);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (lane == 0) s_red[warp] = d;
            __syncthreads();
            float dot = 0.f;
            for (int i = 0; i < FZ_THREADS / 32; ++i) dot += s_red[i];
            g = 1.0f / (1.0f + expf(-dot));
        }
        __syncthreads();

        for (int v = tid; v < vec; v += FZ_THREADS) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            for (int j = 0; j < k; ++j) {
                const int64_t r = s_row[j];
                if (r < 0) continue;
                float f[8];
                unpack8(__ldg(reinterpret_cast<const uint4*>(y + r * H) + v), f);
                const float wj = s_w[j];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
            }
            if (y_sh) {
                float f[8];
                unpack8(__ldg(reinterpret_cast<const uint4*>(y_sh + t * H) + v), f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            reinterpret_cast<uint4*>(out + t * H)[v] = o;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_finalize(const FinalizeLaunch& L, int num_sms, cudaStream_t s) {
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(L.T, (int64_t)num_sms * 16));
    finalize_kernel<<<grid, FZ_THREADS, 0, s>>>(L.y, L.rows_cap, L.pair_row, L.w, L.T, L.k, L.H, L.y_sh, L.x,
                                                L.gate_w, L.out, L.hdr ? &L.hdr->status : nullptr);
    return cudaGetLastError();
}

}  // namespace moe
