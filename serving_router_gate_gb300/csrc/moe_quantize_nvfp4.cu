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
// With power-of-two row scales the per-element division is replaced by a product
// with the block's rounded reciprocal and one exact residual correction, which
// provably gives the division's codes (quantize_block).  A row may also be written
// to several destination rows (a token row to the rows of its routed pairs).
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

// A group of G threads per row (G = 32, 64, 128 or 256; 256 / G rows per CTA
// round).  A row is read in chunks of G * CB blocks: thread i of the group holds
// blocks i, i + G, ... of the chunk, two 16-byte loads each.  The row maximum is an
// unsigned maximum of the bf16 patterns with the sign cleared, reduced by shuffles
// (and through shared memory when the group spans several warps).  A row of one
// chunk stays in registers from the maximum to the codes; a longer row is read a
// second time for the codes (the repeat comes from L2).  Many rows: G = 32, CB = 4
// (a warp per row, 4 KB in flight per warp); few rows: one block per thread.
constexpr int Q4_THREADS = 256;

template <int CB>
__device__ __forceinline__ void load_chunk(const uint4* src, int c0, int G, int nblk, int gt, bool live,
                                           uint4 (&v)[CB][2], uint32_t (&bm)[CB]) {
#pragma unroll
    for (int j = 0; j < CB; ++j) {
        const int b = c0 + gt + G * j;
        if (live && b < nblk) {
            v[j][0] = __ldg(src + 2 * b);
            v[j][1] = __ldg(src + 2 * b + 1);
        } else {
            v[j][0] = v[j][1] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int j = 0; j < CB; ++j) bm[j] = absmax_bf16x8(absmax_bf16x8(0u, v[j][0]), v[j][1]);
}

// block scale code and the 16 codes (as 8 bytes) of one block of values v with
// block maximum bm under row scale s
__device__ __forceinline__ uint2 quantize_block(const uint4 (&v)[2], uint32_t bm, float s, bool pow2,
                                                uint8_t& code) {
    const float bmax = packed_max_to_float(bm);
    code = 0;
    if (s != 0.0f) code = __nv_cvt_float_to_fp8(__fdiv_rn(bmax, __fmul_rn(6.0f, s)), __NV_SATFINITE, __NV_E4M3);
    const float denom = __fmul_rn(e4m3_value(code), s);
    float f[16];
    unpack8(v[0], f);
    unpack8(v[1], f + 8);
    uint32_t w2[2] = {0u, 0u};
    if (denom != 0.0f) {
        const float rcp = __frcp_rn(denom);
        float y[16];
        if (pow2 && denom >= 1.17549435e-38f && rcp >= 1.17549435e-38f && bmax <= 3.40282347e38f) {
            // Power-of-two row scale: denom = sb * 2^e has at most 4 significant bits and
            // every v at most 8, so a quotient v / denom that is not an E2M1 rounding
            // threshold t (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) differs from it by more than
            // 2^-9 relative (v - t * denom is 0 or a multiple of a quantum that large), and
            // one at a threshold is met exactly by y + (v - y denom) / denom, y = v * rn(1 /
            // denom) (the residual is exact).  Either way the code equals that of the
            // binary32 quotient, with no division.
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float y0 = __fmul_rn(f[i], rcp);
                y[i] = fmaf(fmaf(-y0, denom, f[i]), rcp, y0);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(f[i], denom);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) w2[i >> 2] |= e2m1x2(y[2 * i], y[2 * i + 1]) << (8 * (i & 3));
    }
    return make_uint2(w2[0], w2[1]);
}

template <int CB>
__global__ void __launch_bounds__(Q4_THREADS) quantize_nvfp4_rows_kernel(const __grid_constant__ Nvfp4QuantSeg seg0,
                                                                        const __grid_constant__ Nvfp4QuantSeg seg1,
                                                                        int nseg, int G) {
    __shared__ uint32_t red[Q4_THREADS / 32];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rpc = Q4_THREADS / G;             // rows per CTA round
    const int gi = tid / G, gt = tid - gi * G;  // this thread's group and place in it
    const int w0 = gi * (G / 32), nwg = G / 32;  // the group's warps
    for (int sidx = 0; sidx < nseg; ++sidx) {
        const Nvfp4QuantSeg& sg = sidx == 0 ? seg0 : seg1;
        int64_t rows = sg.rows;
        if (sg.rows_dev) rows = min(rows, (int64_t)max(0, *sg.rows_dev));
        const int K = sg.K;
        const int nblk = K / 16;
        const int sfw = nvfp4_sf_row_bytes(K);
        const int chunk = G * CB;
        // every thread runs the same number of row rounds, so each barrier is reached by
        // the whole CTA
        for (int64_t r0 = (int64_t)blockIdx.x * rpc; r0 < rows; r0 += (int64_t)gridDim.x * rpc) {
            const int64_t r = r0 + gi;
            const bool live = gi < rpc && r < rows;
            const uint4* src = reinterpret_cast<const uint4*>(sg.src + (live ? r : 0) * K);
            uint4 v[CB][2];
            uint32_t bm[CB];
            uint32_t pm = 0;
            for (int c0 = 0; c0 < nblk; c0 += chunk) {
                load_chunk<CB>(src, c0, G, nblk, gt, live, v, bm);
#pragma unroll
                for (int j = 0; j < CB; ++j) pm = __vmaxu2(pm, bm[j]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) pm = __vmaxu2(pm, __shfl_xor_sync(0xffffffffu, pm, off));
            if (G > 32) {
                if (lane == 0) red[warp] = pm;
                __syncthreads();
                pm = 0;
                for (int w = 0; w < nwg; ++w) pm = __vmaxu2(pm, red[w0 + w]);
                __syncthreads();  // red is rewritten in the next round
            }
            if (!live) continue;
            const float amax = packed_max_to_float(pm);
            const float s = sg.pow2 ? pow2_row_scale(amax) : __fdiv_rn(amax, 2688.0f);
            // destinations: row r of q / sb / scale (if given) and, with pair_row, the rows
            // of row r's pairs in q2 / sb2 / scale2 (lane j < k holds pair j's row)
            int32_t prow = -1;
            if (sg.pair_row && lane < sg.k) {
                prow = sg.pair_row[r * sg.k + lane];
                if (prow >= sg.dst2_rows) prow = -1;
            }
            const int nk = sg.pair_row ? sg.k : 0;
            if (gt == 0 && sg.q) sg.scale[r] = s;
            if (gt < nk && prow >= 0) sg.scale2[prow] = s;
            for (int c0 = 0; c0 < nblk; c0 += chunk) {
                if (nblk > chunk) load_chunk<CB>(src, c0, G, nblk, gt, true, v, bm);  // else still in registers
#pragma unroll
                for (int j = 0; j < CB; ++j) {
                    const int b = c0 + gt + G * j;
                    const bool ok = b < nblk;
                    uint8_t code = 0;
                    uint2 qv = make_uint2(0u, 0u);
                    if (ok) qv = quantize_block(v[j], bm[j], s, sg.pow2 != 0, code);
                    if (ok && sg.q) {
                        sg.sb[r * sfw + b] = code;
                        reinterpret_cast<uint2*>(sg.q + r * (K / 2))[b] = qv;
                    }
                    for (int d = 0; d < nk; ++d) {  // every lane takes part in the shuffles
                        const int32_t pr = __shfl_sync(0xffffffffu, prow, d);
                        if (ok && pr >= 0) {
                            sg.sb2[(int64_t)pr * sfw + b] = code;
                            reinterpret_cast<uint2*>(sg.q2 + (int64_t)pr * (K / 2))[b] = qv;
                        }
                    }
                }
            }
            // padding of the block-scale rows
            for (int b0 = nblk; b0 < sfw; b0 += G) {
                const int b = b0 + gt;
                if (b < sfw && sg.q) sg.sb[r * sfw + b] = 0;
                for (int d = 0; d < nk; ++d) {
                    const int32_t pr = __shfl_sync(0xffffffffu, prow, d);
                    if (b < sfw && pr >= 0) sg.sb2[(int64_t)pr * sfw + b] = 0;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize_nvfp4_rows(const Nvfp4QuantSeg* seg, int nseg, int num_sms, cudaStream_t s) {
    if (nseg < 1 || nseg > 2) return cudaErrorInvalidValue;
    int64_t rows = 0, blocks = 0;
    int nblk_max = 0;
    for (int i = 0; i < nseg; ++i) {
        if (seg[i].K <= 0 || seg[i].K % 16 != 0 || seg[i].k < 0 || seg[i].k > 32) return cudaErrorInvalidValue;
        if (!seg[i].q && !seg[i].pair_row) return cudaErrorInvalidValue;
        rows = std::max<int64_t>(rows, seg[i].rows);
        blocks += seg[i].rows * (seg[i].K / 16);
        nblk_max = std::max(nblk_max, seg[i].K / 16);
    }
    if (rows <= 0) return cudaSuccess;
    const Nvfp4QuantSeg empty = seg[0];
    // enough blocks for four per thread on two CTAs per SM: a warp per row; else spread
    // each row over up to 256 threads, one block each
    if (blocks >= (int64_t)num_sms * 2 * Q4_THREADS * 4) {
        const int G = 32;
        const int64_t ctas = (rows + Q4_THREADS / G - 1) / (Q4_THREADS / G);
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)num_sms * 8));
        return launch_k("quantize_nvfp4_rows", quantize_nvfp4_rows_kernel<4>, dim3(grid), dim3(Q4_THREADS), 0, s,
                        seg[0], nseg > 1 ? seg[1] : empty, nseg, G);
    }
    int G = 32;  // a power of two, so that the groups tile the CTA
    while (G < Q4_THREADS && G < nblk_max) G *= 2;
    const int64_t ctas = (rows + Q4_THREADS / G - 1) / (Q4_THREADS / G);
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)num_sms * 8));
    return launch_k("quantize_nvfp4_rows", quantize_nvfp4_rows_kernel<1>, dim3(grid), dim3(Q4_THREADS), 0, s,
                    seg[0], nseg > 1 ? seg[1] : empty, nseg, G);
}

}  // namespace moe
