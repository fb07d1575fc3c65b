// moe_quantize_nvfp4.cu -- NVFP4 quantisation of expert weights and of expert
// activations, rows at a time.
//
// The TensorRT-LLM AutoDeploy MoE PR #10985 (review of torch_moe.py) names NVFP4
// paths of the MoE ops and defines no encoding.  Reading: E2M1 elements, one
// E4M3 scale per 16 consecutive elements of a row, one fp32 scale per row.
// For a row with largest magnitude amax the row scale is s = amax / 2688 (one
// binary32 division; 2688 = 6 * 448) -- or, for activations, the power of two
// s = 2^e with e the smallest integer >= -126 such that amax <= 2688 * 2^e.
// Each block b of 16 elements gets sb = e4m3(bmax / (6 s)) (the product and the
// division in binary32, to nearest with ties to even, saturating at 448), and
// each element q = e2m1(v / (sb * s)) (the product and the division in
// binary32, to nearest with ties to the even code, saturating at 6).  An
// all-zero row gets s = 0 (weights) and zero scales and codes; a block whose
// scale rounds to zero gets zero codes.
//
// Layout written: codes [rows][K/2] bytes, element 2i in the low nibble of byte
// i and 2i + 1 in the high one; block scales [rows][SFW] bytes with
// SFW = 16 * ceil(K / 256) (blocks past K/16 are zero: a row of block scales is
// a whole number of 16-byte pieces, one per 256 elements, the unit a GEMM
// pipeline stage reads); row scales [rows] fp32.
//
// A group of threads per row: each thread loads whole blocks (two 16-byte loads
// of 16 values), the row maximum is an unsigned maximum of the bf16 patterns
// with the sign cleared (reduced over the group), then each thread writes its
// blocks' scales and codes (16 codes as 8 bytes).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t absmax_bf16x8(uint32_t m, const uint4& v) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    return __vmaxu2(m, v.w & 0x7FFF7FFFu);
}

__device__ __forceinline__ float packed_max_to_float(uint32_t m) {
    const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
    return __uint_as_float((hi > lo ? hi : lo) << 16);
}

// the power of two 2^e, e the smallest integer >= -126 with amax <= 2688 * 2^e:
// with amax = f * 2^E (1 <= f < 2) and 2688 = 1.3125 * 2^11, e = E - 11 when
// f <= 1.3125, else E - 10
__device__ __forceinline__ float pow2_row_scale(float amax) {
    const uint32_t b = __float_as_uint(amax);
    int e = (int)(b >> 23) - 127 - 11 + ((b & 0x7FFFFFu) > 0x280000u ? 1 : 0);
    if (e < -126) e = -126;
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

__device__ __forceinline__ float e4m3_value(uint8_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
    return __half2float(__half(h));
}

// two values -> two E2M1 codes in one byte (the first in the low nibble)
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}

// A group of G threads per row (G the row's block count rounded up to a multiple
// of 32, at most 256; 256 / G rows per CTA): thread i of a group holds blocks
// i, i + G, ... of its row in registers (up to Q4_MAXB of them), so a single pass
// over global memory gives the row maximum (reduced over the group's warps), the
// block scales and the codes.  Every thread runs the same number of row rounds, so
// every barrier is reached by the whole CTA.
constexpr int Q4_THREADS = 256;
constexpr int Q4_MAXB = 4;  // blocks per thread: rows of up to 4 * 256 * 16 = 16384 elements

__global__ void __launch_bounds__(Q4_THREADS) quantize_nvfp4_rows_kernel(const __grid_constant__ Nvfp4QuantSeg seg0,
                                                                        const __grid_constant__ Nvfp4QuantSeg seg1,
                                                                        int nseg) {
    __shared__ uint32_t red[Q4_THREADS / 32];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int sidx = 0; sidx < nseg; ++sidx) {
        const Nvfp4QuantSeg& sg = sidx == 0 ? seg0 : seg1;
        int64_t rows = sg.rows;
        if (sg.rows_dev) rows = min(rows, (int64_t)max(0, *sg.rows_dev));
        const int K = sg.K;
        const int nblk = K / 16;
        const int sfw = nvfp4_sf_row_bytes(K);
        const int G = min(Q4_THREADS, (nblk + 31) / 32 * 32);  // threads per row
        const int rpc = Q4_THREADS / G;                        // rows per CTA round
        const int gi = tid / G, gt = tid - gi * G;             // this thread's group and place in it
        const int w0 = gi * (G / 32), nwg = G / 32;            // the group's warps
        for (int64_t r0 = (int64_t)blockIdx.x * rpc; r0 < rows; r0 += (int64_t)gridDim.x * rpc) {
            const int64_t r = r0 + gi;
            const bool live = gi < rpc && r < rows;
            const uint4* src = reinterpret_cast<const uint4*>(sg.src + (live ? r : 0) * K);
            uint4 v[Q4_MAXB][2];
            uint32_t bm[Q4_MAXB];
            uint32_t pm = 0;
#pragma unroll
            for (int j = 0; j < Q4_MAXB; ++j) {
                const int b = gt + j * G;
                bm[j] = 0;
                if (live && b < nblk) {
                    v[j][0] = __ldg(src + 2 * b);
                    v[j][1] = __ldg(src + 2 * b + 1);
                    bm[j] = absmax_bf16x8(absmax_bf16x8(0u, v[j][0]), v[j][1]);
                    pm = __vmaxu2(pm, bm[j]);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) pm = __vmaxu2(pm, __shfl_xor_sync(0xffffffffu, pm, off));
            if (lane == 0) red[warp] = pm;
            __syncthreads();
            pm = 0;
            for (int w = 0; w < nwg; ++w) pm = __vmaxu2(pm, red[min(w0 + w, Q4_THREADS / 32 - 1)]);
            __syncthreads();  // red is rewritten in the next round
            if (!live) continue;
            const float amax = packed_max_to_float(pm);
            const float s = sg.pow2 ? pow2_row_scale(amax) : __fdiv_rn(amax, 2688.0f);
            if (gt == 0) sg.scale[r] = s;
            uint8_t* qrow = sg.q + r * (K / 2);
            uint8_t* sbrow = sg.sb + r * sfw;
#pragma unroll
            for (int j = 0; j < Q4_MAXB; ++j) {
                const int b = gt + j * G;
                if (b >= sfw) continue;
                if (b >= nblk) {  // padding of the block-scale row
                    sbrow[b] = 0;
                    continue;
                }
                const float bmax = packed_max_to_float(bm[j]);
                uint8_t code = 0;
                if (s != 0.0f) code = __nv_cvt_float_to_fp8(__fdiv_rn(bmax, __fmul_rn(6.0f, s)), __NV_SATFINITE, __NV_E4M3);
                sbrow[b] = code;
                const float denom = __fmul_rn(e4m3_value(code), s);
                float f[16];
                unpack8(v[j][0], f);
                unpack8(v[j][1], f + 8);
                uint32_t w2[2] = {0u, 0u};
                if (denom != 0.0f) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t byte = e2m1x2(__fdiv_rn(f[2 * i], denom), __fdiv_rn(f[2 * i + 1], denom));
                        w2[i >> 2] |= byte << (8 * (i & 3));
                    }
                }
                *reinterpret_cast<uint2*>(qrow + 8 * b) = make_uint2(w2[0], w2[1]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize_nvfp4_rows(const Nvfp4QuantSeg* seg, int nseg, int num_sms, cudaStream_t s) {
    if (nseg < 1 || nseg > 2) return cudaErrorInvalidValue;
    int64_t rows = 0;
    for (int i = 0; i < nseg; ++i) rows = std::max<int64_t>(rows, seg[i].rows);
    if (rows <= 0) return cudaSuccess;
    for (int i = 0; i < nseg; ++i)
        if (seg[i].K / 16 > Q4_THREADS * Q4_MAXB) return cudaErrorInvalidValue;
    // rows per CTA round of the segment with the most rounds
    int64_t rounds = 1;
    for (int i = 0; i < nseg; ++i) {
        const int nblk = seg[i].K / 16;
        const int rpc = Q4_THREADS / std::min(Q4_THREADS, (nblk + 31) / 32 * 32);
        rounds = std::max<int64_t>(rounds, (seg[i].rows + rpc - 1) / rpc);
    }
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(rounds, (int64_t)num_sms * 8));
    const Nvfp4QuantSeg empty = seg[0];
    return launch_k("quantize_nvfp4_rows", quantize_nvfp4_rows_kernel, dim3(grid), dim3(Q4_THREADS), 0, s, seg[0],
                    nseg > 1 ? seg[1] : empty, nseg);
}

}  // namespace moe
