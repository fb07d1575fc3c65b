// moe_quantize.cu -- row-wise E4M3 quantisation of expert weights and of
// expert activations.
//
// FP8 expert weights (TensorRT-LLM AutoDeploy MoE PR #10985, review of
// torch_moe.py: the MoE ops have FP8 and NVFP4 paths; the pages fix no format).
// Reading: OCP E4M3 with one fp32 scale per output row, scale = amax / 448 and
// q = e4m3(w / scale), both divisions in IEEE binary32, the conversion to
// nearest with ties to even, saturating at 448 (the row's largest |w| maps to
// 448 exactly).  An all-zero row gets scale 0 and q = 0.
//
// One warp per row (grid-stride): a lane-strided max of |w| reduced by a warp
// xor-butterfly (max is exact in any order), then 16-byte loads of 8 bf16
// values and 8-byte stores of their 8 E4M3 bytes.
#include <cuda_fp8.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int QZ_WARPS = 8;

__global__ void __launch_bounds__(QZ_WARPS * 32) quantize_fp8_rows_kernel(const uint16_t* __restrict__ w, int64_t rows,
                                                                         int K, uint8_t* __restrict__ q,
                                                                         float* __restrict__ scale) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int vec = K / 8;
    for (int64_t r = (int64_t)blockIdx.x * QZ_WARPS + (threadIdx.x >> 5); r < rows;
         r += (int64_t)gridDim.x * QZ_WARPS) {
        const uint4* src = reinterpret_cast<const uint4*>(w + r * K);
        float amax = 0.f;
        for (int v = lane; v < vec; v += 32) {
            float f[8];
            unpack8(__ldg(src + v), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float sc = __fdiv_rn(amax, 448.0f);
        if (lane == 0) scale[r] = sc;
        uint2* dst = reinterpret_cast<uint2*>(q + r * K);
        for (int v = lane; v < vec; v += 32) {
            float f[8];
            unpack8(__ldg(src + v), f);
            uint32_t b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                b[i] = sc == 0.f ? 0u
                                 : (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(f[i], sc), __NV_SATFINITE, __NV_E4M3);
            dst[v] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
        }
    }
}

// E4M3 activations (W8A8 experts; same source, same silence on the format).
// Reading: every activation row on its own, scale 2^e with e the smallest
// integer >= -126 such that amax <= 448 * 2^e, q = e4m3(v * 2^-e) to nearest
// with ties to even.  With amax = 1.f * 2^E (1 <= f < 2, binary32 fields) and
// 448 = 1.75 * 2^8: e = E - 8 when f <= 1.75, else E - 7.  Scaling a bf16 value
// by 2^-e is exact in binary32 except where the result underflows, far below
// E4M3's smallest step, where both roundings give the same zero.
struct ActQuantArgs {
    ActQuantSeg seg[2];
    int nseg;
    int64_t rows0;  // rows of seg[0] (its bound): rows of the launch's index space before seg[1]
    int64_t rows_total;
};

__device__ __forceinline__ int act_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int e = (int)(b >> 23) - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return e < -126 ? -126 : e;
}

__global__ void __launch_bounds__(QZ_WARPS * 32) quantize_act_rows_kernel(const __grid_constant__ ActQuantArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    int64_t lim[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        lim[i] = i < a.nseg ? a.seg[i].rows : 0;
        if (i < a.nseg && a.seg[i].rows_dev) lim[i] = min(lim[i], (int64_t)max(0, __ldg(a.seg[i].rows_dev)));
    }
    for (int64_t gr = (int64_t)blockIdx.x * QZ_WARPS + (threadIdx.x >> 5); gr < a.rows_total;
         gr += (int64_t)gridDim.x * QZ_WARPS) {
        const int si = gr < a.rows0 ? 0 : 1;
        const int64_t r = si ? gr - a.rows0 : gr;
        if (r >= lim[si]) continue;
        const ActQuantSeg& sg = a.seg[si];
        const int vec = sg.K / 8;
        const uint4* src = reinterpret_cast<const uint4*>(sg.src + r * sg.K);
        float amax = 0.f;
        for (int v = lane; v < vec; v += 32) {
            float f[8];
            unpack8(__ldg(src + v), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const int e = act_exponent(amax);
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
        if (lane == 0) sg.scale[r] = __uint_as_float((uint32_t)(127 + e) << 23);
        uint2* dst = reinterpret_cast<uint2*>(sg.dst + r * sg.K);
        for (int v = lane; v < vec; v += 32) {
            float f[8];
            unpack8(__ldg(src + v), f);
            uint32_t b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) b[i] = (uint32_t)__nv_cvt_float_to_fp8(f[i] * inv, __NV_SATFINITE, __NV_E4M3);
            dst[v] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
        }
    }
}

}  // namespace

cudaError_t launch_quantize_act_rows(const ActQuantSeg* seg, int nseg, int num_sms, cudaStream_t s) {
    ActQuantArgs a = {};
    a.nseg = 0;
    for (int i = 0; i < nseg && i < 2; ++i)
        if (seg[i].rows > 0) a.seg[a.nseg++] = seg[i];
    if (a.nseg == 0) return cudaSuccess;
    a.rows0 = a.seg[0].rows;
    a.rows_total = a.rows0 + (a.nseg > 1 ? a.seg[1].rows : 0);
    const int64_t want = (a.rows_total + QZ_WARPS - 1) / QZ_WARPS;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    return launch_k(quantize_act_rows_kernel, dim3(grid), dim3(QZ_WARPS * 32), 0, s, a);
}

cudaError_t launch_quantize_fp8_rows(const uint16_t* w, int64_t rows, int K, uint8_t* q, float* scale, int num_sms,
                                     cudaStream_t s) {
    const int64_t want = (rows + QZ_WARPS - 1) / QZ_WARPS;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    return launch_k(quantize_fp8_rows_kernel, dim3(grid), dim3(QZ_WARPS * 32), 0, s, w, rows, K, q, scale);
}

}  // namespace moe
