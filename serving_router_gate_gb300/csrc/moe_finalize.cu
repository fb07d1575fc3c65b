// moe_finalize.cu -- unpermute and routing-weighted combine of each token's
// k expert outputs, plus the (optionally sigmoid-gated) shared expert.
//
// Method: DeepSpeed PR #6964 (AutoTP for MoE models): the layer output is the
// weighted sum of the outputs of the selected experts, formed once per layer;
// vLLM EP FusedMoE patch, ep_reduce_output: the shared expert's output is added
// to the routed output (out = routed_out + shared_out).  The shared gate
// sigmoid(x . w_s) is the Qwen2-MoE-style scaled shared expert.
//
// One CTA (8 warps) per block of TB <= 8 consecutive tokens, grid-stride over
// blocks.  Per block:
//   1. the tokens' pair rows and weights go to shared memory (row -1 = pair
//      skipped; a row outside [-1, rows_cap) is reported and skipped);
//   2. warp w computes the shared gate g of token w: a lane-strided fp32
//      partial dot x . w_s, then a warp xor-butterfly, so every lane holds the
//      same bit-reproducible value;
//   3. the block's TB x H/8 16-byte output vectors are spread over the 256
//      threads, consecutive threads on consecutive vectors of a token; each
//      thread issues the loads of up to 8 pairs' vectors and of the shared
//      expert's vector before using them (with k <= 4 and a bf16 shared row,
//      those of two vectors) and accumulates in fp32 in fixed j order:
//        acc = fma(w_j, y[row_j], acc) for j = 0..k-1 (rows of -1 skipped),
//        acc = fma(g, y_shared, acc), out = bf16_rn(acc),
//      where y_shared is the bf16 shared-expert row or, when the shared FC2 ran
//      with its K split, the fp32 sum of its partial rows in range order.
// TB is picked on the host so that there are at least two blocks per SM when
// the batch allows; with one token (TB = 1) all 256 threads share its row.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int FZ_WARPS = 8;
constexpr int FZ_THREADS = FZ_WARPS * 32;
constexpr int FZ_TB = 8;     // largest token block (one gate warp per token)
constexpr int FZ_MAXK = 32;  // k <= 32
constexpr int FZ_BATCH = 8;  // pair loads issued together

// Each thread takes one output vector at a time and issues the loads of up to
// FZ_BATCH pairs' vectors and of the shared-expert vector before using any.
__global__ void __launch_bounds__(FZ_THREADS, 4) finalize_kernel(
    const uint16_t* __restrict__ y, int64_t rows_cap, const int32_t* __restrict__ pair_row,
    const float* __restrict__ w, int64_t T, int k, int H, int TB, const uint16_t* __restrict__ y_sh,
    const float* __restrict__ y_sh_part, int ksplit, const uint16_t* __restrict__ x,
    const uint16_t* __restrict__ gate_w, uint16_t* __restrict__ out, int32_t* status) {
    __shared__ int32_t s_row[FZ_TB][FZ_MAXK];
    __shared__ float s_w[FZ_TB][FZ_MAXK];
    __shared__ float s_g[FZ_TB];
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int vec = H / 8;
    const bool has_sh = (y_sh != nullptr) || (y_sh_part != nullptr);
    const bool gated = has_sh && (gate_w != nullptr);
    const int64_t nblk = (T + TB - 1) / TB;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t t0 = blk * TB;
        const int nt = (int)min((int64_t)TB, T - t0);
        for (int i = threadIdx.x; i < nt * k; i += FZ_THREADS) {
            const int tt = i / k, j = i - tt * k;
            int32_t r = pair_row[(t0 + tt) * k + j];
            if (r < -1 || (int64_t)r >= rows_cap) {
                report(status, MOE_ERR_DEVICE_BOUNDS);
                r = -1;
            }
            s_row[tt][j] = r;
            s_w[tt][j] = w ? w[(t0 + tt) * k + j] : 1.0f;  // no weights: each kept pair counts once
        }
        if (gated && warp < nt) {
            const uint4* xv = reinterpret_cast<const uint4*>(x + (t0 + warp) * H);
            const uint4* gv = reinterpret_cast<const uint4*>(gate_w);
            float d = 0.f;
#pragma unroll 4
            for (int v = lane; v < vec; v += 32) {
                float a[8], b[8];
                unpack8(__ldg(xv + v), a);
                unpack8(__ldg(gv + v), b);
#pragma unroll
                for (int i = 0; i < 8; ++i) d = fmaf(a[i], b[i], d);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (lane == 0) s_g[warp] = 1.0f / (1.0f + expf(-d));
        }
        __syncthreads();

        const int items = nt * vec;
        if (k <= 4 && !y_sh_part) {
            // k <= 4 and a bf16 shared row (or none): two vectors per thread at a time, the
            // loads of both (their pairs' vectors and shared-expert vectors) in flight
            // before either is used; the shared vectors stay packed until they are added
            for (int f0 = threadIdx.x; f0 < items; f0 += 2 * FZ_THREADS) {
                uint4 ld[2][4], sv[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int f = f0 + u * FZ_THREADS;
                    const bool ok = f < items;
                    const int tt = ok ? f / vec : 0;
                    const int v = ok ? f - tt * vec : 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int32_t r = (ok && b < k) ? s_row[tt][b] : -1;
                        ld[u][b] = r >= 0 ? __ldg(reinterpret_cast<const uint4*>(y + (int64_t)r * H) + v)
                                          : make_uint4(0, 0, 0, 0);
                    }
                    sv[u] = (ok && y_sh) ? __ldg(reinterpret_cast<const uint4*>(y_sh + (t0 + tt) * H) + v)
                                         : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int f = f0 + u * FZ_THREADS;
                    if (f >= items) continue;
                    const int tt = f / vec;
                    const int v = f - tt * vec;
                    float acc[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {  // fixed j order
                        if (b >= k || s_row[tt][b] < 0) continue;
                        const float wj = s_w[tt][b];
                        float fv[8];
                        unpack8(ld[u][b], fv);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, fv[i], acc[i]);
                    }
                    if (has_sh) {
                        const float g = gated ? s_g[tt] : 1.0f;
                        float shf[8];
                        unpack8(sv[u], shf);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, shf[i], acc[i]);
                    }
                    uint4 o;
                    o.x = pack_bf16x2(acc[0], acc[1]);
                    o.y = pack_bf16x2(acc[2], acc[3]);
                    o.z = pack_bf16x2(acc[4], acc[5]);
                    o.w = pack_bf16x2(acc[6], acc[7]);
                    reinterpret_cast<uint4*>(out + (t0 + tt) * H)[v] = o;
                }
            }
        } else {
            for (int f = threadIdx.x; f < items; f += FZ_THREADS) {
                const int tt = f / vec;
                const int v = f - tt * vec;
                float acc[8];
    #pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                float shf[8];
                if (y_sh_part) {
                    // split shared expert: fp32 partials of its K ranges, added in range order
                    const float4* pp = reinterpret_cast<const float4*>(y_sh_part + (t0 + tt) * H) + 2 * v;
                    const int64_t stride = T * (int64_t)H / 4;
                    float4 lo = __ldg(pp), hi = __ldg(pp + 1);
                    for (int q = 1; q < ksplit; ++q) {
                        const float4 a = __ldg(pp + q * stride), b = __ldg(pp + q * stride + 1);
                        lo.x += a.x; lo.y += a.y; lo.z += a.z; lo.w += a.w;
                        hi.x += b.x; hi.y += b.y; hi.z += b.z; hi.w += b.w;
                    }
                    shf[0] = lo.x; shf[1] = lo.y; shf[2] = lo.z; shf[3] = lo.w;
                    shf[4] = hi.x; shf[5] = hi.y; shf[6] = hi.z; shf[7] = hi.w;
                } else if (y_sh) {
                    unpack8(__ldg(reinterpret_cast<const uint4*>(y_sh + (t0 + tt) * H) + v), shf);
                }
                for (int j0 = 0; j0 < k; j0 += FZ_BATCH) {
                    uint4 ld[FZ_BATCH];
                    int32_t rr[FZ_BATCH];
    #pragma unroll
                    for (int b = 0; b < FZ_BATCH; ++b) {
                        const int j = j0 + b;
                        rr[b] = j < k ? s_row[tt][j] : -1;
                        ld[b] = rr[b] >= 0 ? __ldg(reinterpret_cast<const uint4*>(y + (int64_t)rr[b] * H) + v)
                                           : make_uint4(0, 0, 0, 0);
                    }
    #pragma unroll
                    for (int b = 0; b < FZ_BATCH; ++b) {
                        if (rr[b] < 0) continue;
                        const float wj = s_w[tt][j0 + b];
                        float fv[8];
                        unpack8(ld[b], fv);
    #pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, fv[i], acc[i]);
                    }
                }
                if (has_sh) {
                    const float g = gated ? s_g[tt] : 1.0f;
    #pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, shf[i], acc[i]);
                }
                uint4 o;
                o.x = pack_bf16x2(acc[0], acc[1]);
                o.y = pack_bf16x2(acc[2], acc[3]);
                o.z = pack_bf16x2(acc[4], acc[5]);
                o.w = pack_bf16x2(acc[6], acc[7]);
                reinterpret_cast<uint4*>(out + (t0 + tt) * H)[v] = o;
            }
        }
        __syncthreads();  // the next block rewrites the shared arrays
    }
}

}  // namespace

cudaError_t launch_finalize(const FinalizeLaunch& L, int num_sms, cudaStream_t s) {
    // largest token block that still leaves two blocks per SM
    int TB = FZ_TB;
    while (TB > 1 && (L.T + TB - 1) / TB < 2LL * num_sms) TB >>= 1;
    const int64_t nblk = (L.T + TB - 1) / TB;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nblk, (int64_t)num_sms * 4));
    return launch_k("finalize", finalize_kernel, dim3(grid), dim3(FZ_THREADS), 0, s, L.y, L.rows_cap, L.pair_row, L.w,
                    L.T, L.k, L.H, TB, L.y_sh, L.y_sh_part, L.y_sh_part ? L.ksplit : 0, L.x, L.gate_w, L.out,
                    L.hdr ? &L.hdr->status : nullptr);
}

}  // namespace moe
