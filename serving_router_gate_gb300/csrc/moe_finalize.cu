// moe_finalize.cu -- unpermute and routing-weighted combine of each token's
// k expert outputs, plus the (optionally sigmoid-gated) shared expert.
//
// Method: DeepSpeed PR #6964 (AutoTP for MoE models): the layer output is the
// weighted sum of the outputs of the selected experts, formed once per layer;
// vLLM EP FusedMoE patch, ep_reduce_output: the shared expert's output is added
// to the routed output (out = routed_out + shared_out).  The shared gate
// sigmoid(x . w_s) is the Qwen2-MoE-style scaled shared expert.
//
// One warp per work unit -- a token's whole row, or (few tokens) a 256-column
// slice of it -- 8 warps per CTA, grid-stride.  Lane j < k holds pair j's row
// and weight and broadcasts them with shuffles.  Each lane owns the 16-byte
// vectors lane, lane+32, ... of the unit; it issues the loads of up to 8 pairs'
// rows (and then of the shared-expert row) before using them, and accumulates
// in fp32 in fixed j order:
//   acc = fma(w_j, y[row_j], acc) for j = 0..k-1 (rows of -1 skipped),
//   acc = fma(g, y_shared, acc), out = bf16_rn(acc).
// The gate dot product x . w_s is a per-lane strided partial sum followed by a
// warp xor-butterfly, so every lane holds the same bit-reproducible value.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int FZ_WARPS = 8;

// FZ_UNROLL vectors per lane per pass; FZ_BATCH pairs whose loads are issued
// together (rows: 2 x 4; slices, one vector per lane: 1 x 8)
template <int FZ_UNROLL, int FZ_BATCH>
__global__ void __launch_bounds__(FZ_WARPS * 32, 3) finalize_kernel(
    const uint16_t* __restrict__ y, int64_t rows_cap, const int32_t* __restrict__ pair_row,
    const float* __restrict__ w, int64_t T, int k, int H, int unit_cols, const uint16_t* __restrict__ y_sh,
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gate_w, uint16_t* __restrict__ out,
    int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int vec = H / 8;
    const int units_per_token = H / unit_cols;
    const int64_t units = T * units_per_token;
    for (int64_t un = (int64_t)blockIdx.x * FZ_WARPS + warp; un < units; un += (int64_t)gridDim.x * FZ_WARPS) {
        const int64_t t = un / units_per_token;
        const int v_beg = (int)(un % units_per_token) * (unit_cols / 8);
        const int v_end = v_beg + unit_cols / 8;
        int64_t my_row = -1;
        float my_w = 0.f;
        if (lane < k) {
            const int32_t r = pair_row[t * k + lane];
            my_row = r;
            if (r < -1 || (int64_t)r >= rows_cap) {
                report(status, MOE_ERR_DEVICE_BOUNDS);
                my_row = -1;
            }
            my_w = w[t * k + lane];
        }
        float g = 1.0f;
        if (y_sh && gate_w) {
            const uint4* xv = reinterpret_cast<const uint4*>(x + t * H);
            const uint4* gv = reinterpret_cast<const uint4*>(gate_w);
            float d = 0.f;
            for (int v = lane; v < vec; v += 32) {
                float a[8], b[8];
                unpack8(__ldg(xv + v), a);
                unpack8(__ldg(gv + v), b);
#pragma unroll
                for (int i = 0; i < 8; ++i) d = fmaf(a[i], b[i], d);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            g = 1.0f / (1.0f + expf(-d));
        }
        uint4* orow = reinterpret_cast<uint4*>(out + t * H);
        const uint4* srow = y_sh ? reinterpret_cast<const uint4*>(y_sh + t * H) : nullptr;
        for (int v0 = v_beg + lane; v0 < v_end; v0 += 32 * FZ_UNROLL) {
            float acc[FZ_UNROLL][8];
#pragma unroll
            for (int u = 0; u < FZ_UNROLL; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
            // pairs in batches of FZ_BATCH: every load of a batch is issued before any use
            for (int j0 = 0; j0 < k; j0 += FZ_BATCH) {
                uint4 ld[FZ_BATCH][FZ_UNROLL];
                float wj[FZ_BATCH];
#pragma unroll
                for (int b = 0; b < FZ_BATCH; ++b) {
                    const int j = j0 + b;
                    const int64_t r = __shfl_sync(0xffffffffu, my_row, j & 31);
                    wj[b] = __shfl_sync(0xffffffffu, my_w, j & 31);
                    const bool use = (j < k) && (r >= 0);
                    if (!use) wj[b] = 0.f;
                    const uint4* yrow = reinterpret_cast<const uint4*>(y + (use ? r : 0) * H);
#pragma unroll
                    for (int u = 0; u < FZ_UNROLL; ++u) {
                        const int v = v0 + 32 * u;
                        ld[b][u] = (use && v < v_end) ? __ldg(yrow + v) : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int b = 0; b < FZ_BATCH; ++b) {
                    if (j0 + b >= k) break;
                    if (__shfl_sync(0xffffffffu, my_row, (j0 + b) & 31) < 0) continue;
#pragma unroll
                    for (int u = 0; u < FZ_UNROLL; ++u) {
                        float f[8];
                        unpack8(ld[b][u], f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[u][i] = fmaf(wj[b], f[i], acc[u][i]);
                    }
                }
            }
            if (srow) {
                uint4 ld[FZ_UNROLL];
#pragma unroll
                for (int u = 0; u < FZ_UNROLL; ++u) {
                    const int v = v0 + 32 * u;
                    ld[u] = v < v_end ? __ldg(srow + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < FZ_UNROLL; ++u) {
                    float f[8];
                    unpack8(ld[u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[u][i] = fmaf(g, f[i], acc[u][i]);
                }
            }
#pragma unroll
            for (int u = 0; u < FZ_UNROLL; ++u) {
                const int v = v0 + 32 * u;
                if (v < v_end) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                    o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                    o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                    o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                    orow[v] = o;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_finalize(const FinalizeLaunch& L, int num_sms, cudaStream_t s) {
    // work unit of one warp: a whole row when there are enough tokens to fill
    // the GPU, else 256-column slices (each slice recomputes the gate dot)
    int unit_cols = L.H;
    if (L.T < 64LL * num_sms && L.H % 256 == 0) unit_cols = 256;
    const int64_t units = L.T * (L.H / unit_cols);
    const int64_t want = (units + FZ_WARPS - 1) / FZ_WARPS;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    if (unit_cols == L.H)
        return launch_k(finalize_kernel<2, 4>, dim3(grid), dim3(FZ_WARPS * 32), 0, s, L.y, L.rows_cap, L.pair_row,
                        L.w, L.T, L.k, L.H, unit_cols, L.y_sh, L.x, L.gate_w, L.out,
                        L.hdr ? &L.hdr->status : nullptr);
    return launch_k(finalize_kernel<1, 8>, dim3(grid), dim3(FZ_WARPS * 32), 0, s, L.y, L.rows_cap, L.pair_row, L.w,
                    L.T, L.k, L.H, unit_cols, L.y_sh, L.x, L.gate_w, L.out, L.hdr ? &L.hdr->status : nullptr);
}

}  // namespace moe
