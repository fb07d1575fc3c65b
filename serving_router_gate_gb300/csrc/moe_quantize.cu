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
#include <mutex>

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
};

__device__ __forceinline__ int act_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int e = (int)(b >> 23) - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return e < -126 ? -126 : e;
}

// One CTA of 256 threads quantises a group of R = 4 / VPT consecutive rows at a
// time, each thread owning VPT 16-byte vectors (8 bf16) of every one of those
// rows.  The vectors arrive by cp.async in a double-buffered shared-memory
// staging area: the copies of the next group are issued before the current one
// is reduced and stored, and each thread reads back only its own vectors (no
// barrier besides the reduction's).  Rows longer than 256 * 4 * 8 values take a
// two-pass loop instead.
constexpr int QA_THREADS = 256;
constexpr int QA_WARPS = QA_THREADS / 32;
constexpr int QA_VEC = 4;  // 16-byte vectors per thread per row group

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// four values scaled by inv (a power of two) -> four E4M3 bytes, two per conversion
__device__ __forceinline__ uint32_t e4m3x4(const float* f, float inv) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[0] * inv, f[1] * inv), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[2] * inv, f[3] * inv), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// |v| of a finite bf16 value orders like its bit pattern with the sign cleared,
// so a row's amax is an unsigned maximum of those 15-bit patterns (two per word)
__device__ __forceinline__ uint32_t absmax_bf16x8(uint32_t m, const uint4& v) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    return __vmaxu2(m, v.w & 0x7FFF7FFFu);
}

// amax over the CTA for each of the R rows (packed per-thread maxima in, binary32
// amax out); red: [R][QA_WARPS] shared words
template <int R>
__device__ __forceinline__ void block_amax(const uint32_t (&pk)[R], float (&am)[R], uint32_t* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, max(pk[rr] & 0xFFFFu, pk[rr] >> 16));
        if (lane == 0) red[rr * QA_WARPS + warp] = m;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        uint32_t m = red[rr * QA_WARPS];
#pragma unroll
        for (int w = 1; w < QA_WARPS; ++w) m = max(m, red[rr * QA_WARPS + w]);
        am[rr] = __uint_as_float(m << 16);
    }
    __syncthreads();  // red is rewritten by the next group
}

// The codes of source row `row` (vector j of this thread: q[j]) and its scale go
// to row `row` of dst and, with pair_row, to each pair row of dst2.
template <int VPT>
__device__ __forceinline__ void store_row(const ActQuantSeg& sg, int64_t row, const uint2 (&q)[VPT], float scale) {
    const int vec = sg.K / 8;
    if (sg.dst) {
        if (threadIdx.x == 0) sg.scale[row] = scale;
        uint2* dst = reinterpret_cast<uint2*>(sg.dst + row * sg.K);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int idx = threadIdx.x + j * QA_THREADS;
            if (idx < vec) dst[idx] = q[j];
        }
    }
    if (sg.pair_row) {
        for (int jj = 0; jj < sg.k; ++jj) {
            const int32_t r = __ldg(sg.pair_row + row * sg.k + jj);
            if (r < 0 || (int64_t)r >= sg.dst2_rows) continue;
            if (threadIdx.x == 0) sg.scale2[r] = scale;
            uint2* dst = reinterpret_cast<uint2*>(sg.dst2 + (int64_t)r * sg.K);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int idx = threadIdx.x + j * QA_THREADS;
                if (idx < vec) dst[idx] = q[j];
            }
        }
    }
}

// stage[buf][i * QA_THREADS + thread]: vector i = rr * VPT + j of the group
template <int VPT>
__device__ __forceinline__ void issue_group(uint4* stage, const ActQuantSeg& sg, int64_t base, int64_t lim) {
    constexpr int R = QA_VEC / VPT;
    const int vec = sg.K / 8;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int64_t row = base + rr;
        const uint4* src = reinterpret_cast<const uint4*>(sg.src + (row < lim ? row : 0) * sg.K);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int idx = threadIdx.x + j * QA_THREADS;
            cp_async16(stage + (rr * VPT + j) * QA_THREADS + threadIdx.x, src + (idx < vec ? idx : 0),
                       row < lim && idx < vec);
        }
    }
    cp_async_commit();
}

template <int VPT>
__device__ __forceinline__ void quantize_rows_staged(const ActQuantSeg& sg, int64_t lim, uint32_t* red, uint4* stage,
                                                     int cta) {
    constexpr int R = QA_VEC / VPT;
    const int vec = sg.K / 8;
    const int64_t stride = (int64_t)gridDim.x * R;
    int64_t base = (int64_t)cta * R;
    if (base >= lim) return;
    issue_group<VPT>(stage, sg, base, lim);
    for (int it = 0; base < lim; base += stride, ++it) {
        uint4* cur = stage + (it & 1) * QA_VEC * QA_THREADS;
        uint4* nxt = stage + ((it & 1) ^ 1) * QA_VEC * QA_THREADS;
        if (base + stride < lim)
            issue_group<VPT>(nxt, sg, base + stride, lim);
        else
            cp_async_commit();  // an empty group keeps the wait count uniform
        cp_async_wait_one();    // this thread's copies of the current group have landed
        uint4 v[R][VPT];
        uint32_t pk[R];
        float am[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            pk[rr] = 0u;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                v[rr][j] = cur[(rr * VPT + j) * QA_THREADS + threadIdx.x];
                pk[rr] = absmax_bf16x8(pk[rr], v[rr][j]);
            }
        }
        block_amax<R>(pk, am, red);
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int64_t row = base + rr;
            if (row < lim) {
                const int e = act_exponent(am[rr]);
                const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
                uint2 q[VPT];
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    float f[8];
                    unpack8(v[rr][j], f);
                    q[j] = make_uint2(e4m3x4(f, inv), e4m3x4(f + 4, inv));
                }
                store_row<VPT>(sg, row, q, __uint_as_float((uint32_t)(127 + e) << 23));
            }
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// long rows (more than 8192 values): one row per CTA iteration, read twice (amax,
// then quantise)
__device__ __forceinline__ void quantize_rows_loop(const ActQuantSeg& sg, int64_t lim, uint32_t* red, int cta) {
    const int vec = sg.K / 8;
    for (int64_t row = cta; row < lim; row += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(sg.src + row * sg.K);
        uint32_t pk[1] = {0u};
        float am[1];
        for (int idx = threadIdx.x; idx < vec; idx += QA_THREADS) pk[0] = absmax_bf16x8(pk[0], __ldg(src + idx));
        block_amax<1>(pk, am, red);
        const int e = act_exponent(am[0]);
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
        const float sc = __uint_as_float((uint32_t)(127 + e) << 23);
        if (threadIdx.x == 0) {
            if (sg.dst) sg.scale[row] = sc;
            if (sg.pair_row)
                for (int jj = 0; jj < sg.k; ++jj) {
                    const int32_t r = __ldg(sg.pair_row + row * sg.k + jj);
                    if (r >= 0 && (int64_t)r < sg.dst2_rows) sg.scale2[r] = sc;
                }
        }
        for (int idx = threadIdx.x; idx < vec; idx += QA_THREADS) {
            float f[8];
            unpack8(__ldg(src + idx), f);
            const uint2 q = make_uint2(e4m3x4(f, inv), e4m3x4(f + 4, inv));
            if (sg.dst) reinterpret_cast<uint2*>(sg.dst + row * sg.K)[idx] = q;
            if (sg.pair_row)
                for (int jj = 0; jj < sg.k; ++jj) {
                    const int32_t r = __ldg(sg.pair_row + row * sg.k + jj);
                    if (r >= 0 && (int64_t)r < sg.dst2_rows)
                        reinterpret_cast<uint2*>(sg.dst2 + (int64_t)r * sg.K)[idx] = q;
                }
        }
    }
}

__global__ void __launch_bounds__(QA_THREADS) quantize_act_rows_kernel(const __grid_constant__ ActQuantArgs a) {
    __shared__ uint32_t red[QA_VEC * QA_WARPS];
    __shared__ uint4 stage[2 * QA_VEC * QA_THREADS];  // 32 KB: two row groups
    pdl_wait();
    pdl_trigger();
    for (int si = 0; si < a.nseg; ++si) {
        const ActQuantSeg& sg = a.seg[si];
        int64_t lim = sg.rows;
        if (sg.rows_dev) lim = min(lim, (int64_t)max(0, __ldg(sg.rows_dev)));
        const int vpt = (sg.K / 8 + QA_THREADS - 1) / QA_THREADS;
        // the second row set starts from the last CTA, so small launches run both at once
        const int cta = si ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
        if (vpt <= 1)
            quantize_rows_staged<1>(sg, lim, red, stage, cta);
        else if (vpt <= 2)
            quantize_rows_staged<2>(sg, lim, red, stage, cta);
        else if (vpt <= 4)
            quantize_rows_staged<4>(sg, lim, red, stage, cta);
        else
            quantize_rows_loop(sg, lim, red, cta);
    }
}

}  // namespace

cudaError_t launch_quantize_act_rows(const ActQuantSeg* seg, int nseg, int num_sms, cudaStream_t s) {
    ActQuantArgs a = {};
    a.nseg = 0;
    for (int i = 0; i < nseg && i < 2; ++i)
        if (seg[i].rows > 0) a.seg[a.nseg++] = seg[i];
    if (a.nseg == 0) return cudaSuccess;
    // one CTA per row group of the two row sets together, at most one wave of
    // resident CTAs (several per SM: 32 KB of staging each, so the largest
    // shared-memory carve-out)
    static std::once_flag once;
    static int per_sm = 1;
    std::call_once(once, [] {
        cudaFuncSetAttribute(quantize_act_rows_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_act_rows_kernel, QA_THREADS, 0) ==
                cudaSuccess &&
            n > 0)
            per_sm = n;
    });
    int64_t want = 0;
    for (int i = 0; i < a.nseg; ++i) {
        const int vpt = (a.seg[i].K / 8 + QA_THREADS - 1) / QA_THREADS;
        const int R = vpt <= 1 ? 4 : vpt <= 2 ? 2 : 1;
        want += (a.seg[i].rows + R - 1) / R;
    }
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * per_sm));
    return launch_k("quantize_act_rows", quantize_act_rows_kernel, dim3(grid), dim3(QA_THREADS), 0, s, a);
}

cudaError_t launch_quantize_fp8_rows(const uint16_t* w, int64_t rows, int K, uint8_t* q, float* scale, int num_sms,
                                     cudaStream_t s) {
    const int64_t want = (rows + QZ_WARPS - 1) / QZ_WARPS;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    return launch_k("quantize_fp8_rows", quantize_fp8_rows_kernel, dim3(grid), dim3(QZ_WARPS * 32), 0, s, w, rows, K,
                    q, scale);
}

}  // namespace moe
