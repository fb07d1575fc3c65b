// moe_router.cu -- router of the MoE layer: fp32 gate GEMM on CUDA cores,
// softmax over all experts, certified top-k (ties to the lower expert id),
// optional renormalisation.
//
// Method: vLLM EP FusedMoE patch (ep_fused_moe_patch.py), module docstring
// "EP expert dispatch" -- top-k routing yields global expert ids, the same on
// every rank -- and its patched __init__ (renormalize defaults to true; routing
// over the global expert count).  The softmax runs over all experts before the
// top-k; selection is by logit (softmax is monotone in the logit).
//
// Two kernels:
//  1. router_logits_kernel: partial logits l[t,e] over a K range per CTA.
//     Tile 128 tokens x 64 experts x K-range; each thread owns 8x4 outputs,
//     read from row-major padded shared-memory tiles.  Accumulation is nested (32-term
//     chains per 32-k chunk -> groups of 8 chunks -> the CTA's range), which
//     keeps the worst-case rounding error of every logit below
//     gamma_n * (||x_t|| ||w_e|| + |b_e|) with a small n (about 70 for
//     H = 7168) instead of n = H.  The CTAs of the first token/expert tile
//     also emit the partial squared norms of x rows and Wg rows.
//  2. router_select_kernel: one warp per token.  Sums the split partials in
//     fixed order, adds the bias, and takes the k+1 largest logits (ties ->
//     lower id).  Consecutive candidates whose fp32 gap is within twice the
//     per-token bound form a cluster whose true order fp32 cannot decide; each
//     cluster that touches the top k is recomputed with a compensated fp32
//     dot product (about twice fp32's precision, on the fp32 pipes) and
//     re-ordered; only if those values still leave a gap inside their own
//     bound is the cluster recomputed in fp64 from the exact bf16 x fp32
//     products (ties -> lower id).  Then the fp32
//     softmax (expf) over all E logits, the selected probabilities, and the
//     optional renormalisation (divide by their sum, in j order).
#include <float.h>
#include <limits.h>
#include <stdint.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int RT_BT = 128;       // tokens per CTA
constexpr int RT_BE = 64;        // experts per CTA
constexpr int RT_BK = 32;        // K per shared-memory chunk (level-1 sum length)
constexpr int RT_GROUP = 8;      // chunks per level-2 group
constexpr int RT_THREADS = 256;
constexpr int RT_TARGET_MAX = 2048;  // upper bound on CTAs the split plan aims for
constexpr int RT_MAX_SPLIT = 32;

constexpr int RS_WARPS = 8;      // select: tokens (warps) per CTA

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
    // 16-byte global->shared copy; zero-fills when !valid (source size 0)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Tile: 128 tokens x 64 experts x a K range per CTA, 256 threads, 8 x 4 outputs
// per thread (tokens 4 tg .. 4 tg + 3 and 64 + 4 tg .. + 3, experts eg + 16 j).
// Both operands sit row-major in shared memory in rows padded to 36 floats:
// xs[token][k] (fp32, widened from bf16 once by the thread that stages it) and
// ws[expert][k] (copied as it is by cp.async).  Per 4 k a thread reads its 8 token
// quads and its 4 expert quads with 12 16-byte loads -- a token quad is broadcast to
// half a warp, the 16 expert rows of a warp fall on all 8 bank quads (two wavefronts)
// -- and issues 128 FMAs.  The staging reads are coalesced: per warp instruction 8
// token rows x 64 contiguous bytes, or 4 Wg rows x 128 bytes; the widened token
// pieces go to shared memory as two 16-byte stores that cover all 32 banks per 8
// lanes.  Chunk c is computed from buffer c & 1 while the next chunk's token pieces
// load into registers and its Wg pieces copy into the other buffer; one barrier per
// chunk.  Each logit's sum: per 32-k chunk one chain in ascending k whose first term
// is the rounded product, chunks summed in groups of 8, groups summed over the CTA's
// range -- a rounding depth of 32 + 8 + groups per range.  The expert tiles of one
// token tile are adjacent CTAs, so they share the token rows through L2.  CTAs of
// expert tile 0 also emit the partial squared norms of their token rows, CTAs of
// token tile 0 those of their Wg rows.
constexpr int RT_LD = RT_BK + 4;  // padded row (floats): 144 bytes, 16-byte aligned
// two tile buffers, then the range-level sums of every thread's 32 outputs
constexpr size_t RT_SMEM = sizeof(float) * (2 * RT_LD * (RT_BT + RT_BE) + 32 * RT_THREADS);

__global__ void __launch_bounds__(RT_THREADS, 2) router_logits_kernel(const uint16_t* __restrict__ x,
                                                                      const float* __restrict__ Wg, int64_t T,
                                                                      int H, int E, int KC,
                                                                      float* __restrict__ part,
                                                                      float* __restrict__ xsq,
                                                                      float* __restrict__ wsq) {
    extern __shared__ __align__(16) float rt_smem[];
    pdl_wait();
    pdl_trigger();
    float (*xs)[RT_BT][RT_LD] = reinterpret_cast<float (*)[RT_BT][RT_LD]>(rt_smem);
    float (*ws)[RT_BE][RT_LD] = reinterpret_cast<float (*)[RT_BE][RT_LD]>(rt_smem + 2 * RT_BT * RT_LD);

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * RT_BE;               // expert tiles vary fastest
    const int64_t t0 = (int64_t)blockIdx.y * RT_BT;
    const int sp = blockIdx.z;
    const int kbeg = sp * KC;
    const int kend = min(H, kbeg + KC);
    const int nchunk = (kend - kbeg) / RT_BK;

    // staging: token pieces tid and tid + 256 of a chunk's 512 (token p / 4, k 8 (p % 4)
    // .. + 7, bf16); Wg pieces tid and tid + 256 (expert p / 8, k 4 (p % 8) .. + 3, fp32)
    const int xq = tid & 3;
    const int xt = tid >> 2;                         // tokens xt and xt + 64
    const bool xv0 = t0 + xt < T, xv1 = t0 + xt + 64 < T;
    const uint16_t* xsrc0 = x + (xv0 ? t0 + xt : 0) * (int64_t)H + kbeg + 8 * xq;
    const uint16_t* xsrc1 = x + (xv1 ? t0 + xt + 64 : 0) * (int64_t)H + kbeg + 8 * xq;
    const int wq = tid & 7;
    const int we = tid >> 3;                         // experts we and we + 32
    const bool wv0 = e0 + we < E, wv1 = e0 + we + 32 < E;
    const float* wsrc0 = Wg + (int64_t)(wv0 ? e0 + we : 0) * H + kbeg + 4 * wq;
    const float* wsrc1 = Wg + (int64_t)(wv1 ? e0 + we + 32 : 0) * H + kbeg + 4 * wq;
    const bool wnorm = blockIdx.y == 0;              // this CTA emits the Wg row norms

    uint4 sx0, sx1;                                  // the next chunk's token pieces
    auto load_x = [&](int c) {
        if (c < nchunk) {
            sx0 = xv0 ? __ldg(reinterpret_cast<const uint4*>(xsrc0 + c * RT_BK)) : make_uint4(0, 0, 0, 0);
            sx1 = xv1 ? __ldg(reinterpret_cast<const uint4*>(xsrc1 + c * RT_BK)) : make_uint4(0, 0, 0, 0);
        }
    };
    auto copy_w = [&](int c, int buf) {
        if (c < nchunk) {
            cp_async16(&ws[buf][we][4 * wq], wsrc0 + c * RT_BK, wv0);
            cp_async16(&ws[buf][we + 32][4 * wq], wsrc1 + c * RT_BK, wv1);
        }
        cp_async_commit();
    };
    float nx0 = 0.f, nx1 = 0.f, nw0 = 0.f, nw1 = 0.f;  // partial squared norms (this thread's k)
    auto store_x = [&](int buf) {
        float f[8];
        unpack8(sx0, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) nx0 = fmaf(f[i], f[i], nx0);
        *reinterpret_cast<float4*>(&xs[buf][xt][8 * xq]) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(&xs[buf][xt][8 * xq + 4]) = make_float4(f[4], f[5], f[6], f[7]);
        unpack8(sx1, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) nx1 = fmaf(f[i], f[i], nx1);
        *reinterpret_cast<float4*>(&xs[buf][xt + 64][8 * xq]) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(&xs[buf][xt + 64][8 * xq + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    };

    // compute layout: warp w, lane: expert group eg = lane & 15, token group tg = 2 w + lane / 16
    const int lane = tid & 31, wid = tid >> 5;
    const int eg = lane & 15;
    const int tg = 2 * wid + (lane >> 4);
    // level 3 (the range) lives in shared memory: it changes once per 8 chunks
    float* a3s = rt_smem + 2 * RT_LD * (RT_BT + RT_BE) + tid;  // element q at a3s[q * RT_THREADS]
    float a1[8][4], a2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a2[i][j] = 0.f;
            a3s[(i * 4 + j) * RT_THREADS] = 0.f;
        }

    auto step = [&](int c) {
        const int buf = c & 1;
        load_x(c + 1);
        copy_w(c + 1, buf ^ 1);  // the other buffer was last read by chunk c - 1
        if (wnorm) {
            const float4 p = *reinterpret_cast<const float4*>(&ws[buf][we][4 * wq]);
            const float4 q = *reinterpret_cast<const float4*>(&ws[buf][we + 32][4 * wq]);
            nw0 = fmaf(p.x, p.x, fmaf(p.y, p.y, fmaf(p.z, p.z, fmaf(p.w, p.w, nw0))));
            nw1 = fmaf(q.x, q.x, fmaf(q.y, q.y, fmaf(q.z, q.z, fmaf(q.w, q.w, nw1))));
        }
#pragma unroll
        for (int kq = 0; kq < RT_BK / 4; ++kq) {
            float4 w4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w4[j] = *reinterpret_cast<const float4*>(&ws[buf][eg + 16 * j][4 * kq]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = (i < 4 ? 0 : 64) + 4 * tg + (i & 3);
                const float4 x4 = *reinterpret_cast<const float4*>(&xs[buf][row][4 * kq]);
                const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float wv = kk == 0 ? w4[j].x : kk == 1 ? w4[j].y : kk == 2 ? w4[j].z : w4[j].w;
                        a1[i][j] = (kq == 0 && kk == 0) ? __fmul_rn(xv[kk], wv) : fmaf(xv[kk], wv, a1[i][j]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) a2[i][j] += a1[i][j];
        if ((c % RT_GROUP) == RT_GROUP - 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    a3s[(i * 4 + j) * RT_THREADS] += a2[i][j];
                    a2[i][j] = 0.f;
                }
        }
        if (c + 1 < nchunk) store_x(buf ^ 1);
        cp_async_wait_group<0>();
        __syncthreads();
    };
    load_x(0);
    copy_w(0, 0);
    if (nchunk > 0) store_x(0);
    cp_async_wait_group<0>();
    __syncthreads();
    for (int c = 0; c < nchunk; ++c) step(c);
    float a3[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a3[i][j] = a3s[(i * 4 + j) * RT_THREADS] + a2[i][j];

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t t = t0 + (i < 4 ? 0 : 64) + 4 * tg + (i & 3);
        if (t >= T) continue;
        float* dst = part + ((int64_t)sp * T + t) * E + e0 + eg;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (e0 + eg + 16 * j < E) dst[16 * j] = a3[i][j];
    }
    // squared norms: the 4 lanes of a token row (xq) and the 8 of a Wg row (wq) are
    // adjacent lanes of one warp
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        nx0 += __shfl_xor_sync(0xffffffffu, nx0, off);
        nx1 += __shfl_xor_sync(0xffffffffu, nx1, off);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
        nw0 += __shfl_xor_sync(0xffffffffu, nw0, off);
        nw1 += __shfl_xor_sync(0xffffffffu, nw1, off);
    }
    if (blockIdx.x == 0 && xq == 0) {
        if (xv0) xsq[(int64_t)sp * T + t0 + xt] = nx0;
        if (xv1) xsq[(int64_t)sp * T + t0 + xt + 64] = nx1;
    }
    if (wnorm && wq == 0) {
        if (wv0) wsq[(int64_t)sp * E + e0 + we] = nw0;
        if (wv1) wsq[(int64_t)sp * E + e0 + we + 32] = nw1;
    }
}

// Compensated (doubled-precision) dot product of one bf16 x row with one fp32
// Wg row, by one warp, on the fp32 pipes.  Every product x_h * w_h is split
// exactly into ph + pl (ph = fl(x*w), pl = fma(x, w, -ph)); ph is added to a
// running sum by the error-free TwoSum, whose rounding error joins pl in a
// plain fp32 correction sum (the Dot2 scheme of Ogita, Rump and Oishi,
// "Accurate sum and dot product", 2005).  Lane l keeps four accumulators
// (piece l + 32 j goes to accumulator j mod 4, H/128 products each); the 128
// accumulators are then combined by TwoSum (lanes: xor butterfly, so every lane
// ends with the same pair).  Returned as the fp64 sum hi + lo of the final
// pair, with no rounding to fp32: |result - exact| <= (gamma_{H/128} +
// gamma_128)^2 * sum_h |x_h w_h| (no underflow).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ double refine_dot2(const uint16_t* __restrict__ xrow, const float* __restrict__ wrow, int H, int lane) {
    float hs[4] = {0.f, 0.f, 0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
    const int pieces = H / 8;
    for (int p0 = lane; p0 < pieces; p0 += 128) {
        uint4 xv[4];
        float4 w0[4], w1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = p0 + 32 * i;
            const bool ok = p < pieces;
            xv[i] = ok ? __ldg(reinterpret_cast<const uint4*>(xrow) + p) : make_uint4(0, 0, 0, 0);
            w0[i] = ok ? __ldg(reinterpret_cast<const float4*>(wrow) + 2 * p) : make_float4(0.f, 0.f, 0.f, 0.f);
            w1[i] = ok ? __ldg(reinterpret_cast<const float4*>(wrow) + 2 * p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float xf[8];
            unpack8(xv[i], xf);
            const float wf[8] = {w0[i].x, w0[i].y, w0[i].z, w0[i].w, w1[i].x, w1[i].y, w1[i].z, w1[i].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float ph = __fmul_rn(xf[j], wf[j]);
                const float pl = fmaf(xf[j], wf[j], -ph);
                float sn, e;
                two_sum(hs[i], ph, sn, e);
                hs[i] = sn;
                cs[i] = __fadd_rn(cs[i], __fadd_rn(e, pl));
            }
        }
    }
    float S = hs[0], C = cs[0];
#pragma unroll
    for (int i = 1; i < 4; ++i) {
        float sn, e;
        two_sum(S, hs[i], sn, e);
        S = sn;
        C = __fadd_rn(C, __fadd_rn(e, cs[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oS = __shfl_xor_sync(0xffffffffu, S, off);
        const float oC = __shfl_xor_sync(0xffffffffu, C, off);
        float sn, e;
        two_sum(S, oS, sn, e);  // exact: e = S + oS - sn on both lanes
        S = sn;
        C = __fadd_rn(__fadd_rn(C, oC), e);
    }
    return (double)S + (double)C;
}

// fp64 dot product of one bf16 x row with one fp32 Wg row, by one warp.  Lane
// l takes the 8-element pieces l, l + 32, ... of the row; the loads of four
// pieces are issued together and feed four independent fp64 partial sums
// (piece i into sum i mod 4), added as (s0 + s1) + (s2 + s3) and then summed
// over the lanes by an xor butterfly.  Every lane returns the same value.
// Each bf16 x fp32 product is exact in fp64; the sums' rounding stays within
// gamma_{H+2}(fp64) of the exact dot product (H terms, two more additions).
__device__ double refine_dot(const uint16_t* __restrict__ xrow, const float* __restrict__ wrow, int H, int lane) {
    double s[4] = {0.0, 0.0, 0.0, 0.0};
    const int pieces = H / 8;
    for (int p0 = lane; p0 < pieces; p0 += 128) {
        uint4 xv[4];
        float4 w0[4], w1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = p0 + 32 * i;
            const bool ok = p < pieces;
            xv[i] = ok ? __ldg(reinterpret_cast<const uint4*>(xrow) + p) : make_uint4(0, 0, 0, 0);
            w0[i] = ok ? __ldg(reinterpret_cast<const float4*>(wrow) + 2 * p) : make_float4(0.f, 0.f, 0.f, 0.f);
            w1[i] = ok ? __ldg(reinterpret_cast<const float4*>(wrow) + 2 * p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float xf[8];
            unpack8(xv[i], xf);
            s[i] = fma((double)xf[0], (double)w0[i].x, s[i]);
            s[i] = fma((double)xf[1], (double)w0[i].y, s[i]);
            s[i] = fma((double)xf[2], (double)w0[i].z, s[i]);
            s[i] = fma((double)xf[3], (double)w0[i].w, s[i]);
            s[i] = fma((double)xf[4], (double)w1[i].x, s[i]);
            s[i] = fma((double)xf[5], (double)w1[i].y, s[i]);
            s[i] = fma((double)xf[6], (double)w1[i].z, s[i]);
            s[i] = fma((double)xf[7], (double)w1[i].w, s[i]);
        }
    }
    double t = (s[0] + s[1]) + (s[2] + s[3]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    return t;
}

// Group-limited top-k, group step (warp-wide; every lane returns the same mask).
// Groups are n_group runs of E / n_group consecutive experts; a group's score
// is its largest logit; the topk_group best groups are kept, ties to the lower
// group index.  With fp32 logits within thr/2 of the exact ones, a group whose
// fp32 score lies more than thr above the first dropped group's score is kept
// for certain, one more than thr below the last kept group's is dropped for
// certain.  The groups in between are decided on recomputed scores: the
// experts that can be their maximum (fp32 logit within thr of the group's
// fp32 score) are recomputed with the compensated dot product, and if two of
// those group scores still lie within thr2 of each other, in fp64.
template <int PL>
__device__ __noinline__ uint32_t select_groups(const float (&l)[PL], float* s_l, int* s_cand, double* s_val, int E, int n_group,
                                  int topk_group, float thr, float thr2, const uint16_t* xrow, const float* Wg,
                                  const float* bias, int H, int lane) {
    const int gsize = E / n_group;
#pragma unroll
    for (int i = 0; i < PL; ++i)
        if (lane + 32 * i < E) s_l[lane + 32 * i] = l[i];
    __syncwarp();
    float gm = -INFINITY;  // lane g < n_group: score of group g
    if (lane < n_group)
        for (int e = lane * gsize; e < (lane + 1) * gsize; ++e) gm = fmaxf(gm, s_l[e]);
    // rank the groups: topk_group kept, and the score of the first dropped one
    uint32_t keep = 0;
    float v_last = 0.f, v_next = -INFINITY;
    for (int r = 0; r <= topk_group; ++r) {
        float bv = (lane < n_group && !((keep >> lane) & 1u)) ? gm : -INFINITY;
        int bg = (lane < n_group && !((keep >> lane) & 1u)) ? lane : INT_MAX;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int og = __shfl_xor_sync(0xffffffffu, bg, off);
            if (ov > bv || (ov == bv && og < bg)) {
                bv = ov;
                bg = og;
            }
        }
        if (r < topk_group) {
            keep |= 1u << bg;
            v_last = bv;
        } else {
            v_next = bv;
        }
    }
    if (!(v_last - v_next <= thr)) return keep;  // certified (or no finite competitor)

    // undecided groups: score within [v_next - thr, v_last + thr]
    const float lo = v_next - thr, hi = v_last + thr;
    const bool sure_in = lane < n_group && gm > hi;
    const bool undecided = lane < n_group && !sure_in && gm >= lo;
    const uint32_t und = __ballot_sync(0xffffffffu, undecided);
    const int n_in = __popc(__ballot_sync(0xffffffffu, sure_in));
    const int need = topk_group - n_in;
    // candidates: experts of undecided groups within thr of their group's score
    int nc = 0;
    if (lane == 0) {
        for (int g = 0; g < n_group; ++g) {
            if (!((und >> g) & 1u)) continue;
            float m = -INFINITY;
            for (int e = g * gsize; e < (g + 1) * gsize; ++e) m = fmaxf(m, s_l[e]);
            for (int e = g * gsize; e < (g + 1) * gsize; ++e)
                if (s_l[e] >= m - thr) s_cand[nc++] = e;
        }
    }
    nc = __shfl_sync(0xffffffffu, nc, 0);
    __syncwarp();
    uint32_t result = 0;
    for (int pass = 0; pass < 2; ++pass) {
        for (int c = 0; c < nc; ++c) {
            const int e = s_cand[c];
            double v = pass == 0 ? refine_dot2(xrow, Wg + (int64_t)e * H, H, lane)
                                 : refine_dot(xrow, Wg + (int64_t)e * H, H, lane);
            if (bias) v += (double)bias[e];
            if (lane == 0) s_val[c] = v;
        }
        __syncwarp();
        bool decided = true;
        uint32_t chosen = 0;
        if (lane == 0) {
            // recomputed score of each undecided group, then the need best of them
            double gs[32];
            for (int g = 0; g < n_group; ++g) gs[g] = -INFINITY;
            for (int c = 0; c < nc; ++c) {
                const int g = s_cand[c] / gsize;
                if (s_val[c] > gs[g]) gs[g] = s_val[c];
            }
            double last = 0.0, next = -INFINITY;
            for (int r = 0; r <= need; ++r) {
                int bg = -1;
                for (int g = 0; g < n_group; ++g) {
                    if (!((und >> g) & 1u) || ((chosen >> g) & 1u)) continue;
                    if (bg < 0 || gs[g] > gs[bg]) bg = g;
                }
                if (bg < 0) break;
                if (r < need) {
                    chosen |= 1u << bg;
                    last = gs[bg];
                } else {
                    next = gs[bg];
                }
            }
            decided = pass == 1 || !(last - next <= (double)thr2);
        }
        decided = __shfl_sync(0xffffffffu, decided ? 1 : 0, 0) != 0;
        result = __shfl_sync(0xffffffffu, chosen, 0);
        __syncwarp();
        if (decided) break;
    }
    const uint32_t sure = __ballot_sync(0xffffffffu, sure_in);
    return sure | result;
}

template <int PL>
__device__ __forceinline__ float pick(const float (&l)[PL], int idx) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i)
        if (i == idx) v = l[i];
    return v;
}

// Selection of one token by one warp, from its fp32 logits l (lane holds experts
// lane + 32 i; bias added, NaN already -inf, experts >= E at -inf): the group step
// (if any), the candidates in (logit desc, id asc) order until the cluster that
// holds rank k-1 closes, the certified rechecks of near-tied clusters that touch
// ranks 0..k-1, then the fp32 softmax over all E and the k (renormalised)
// probabilities.  thr / thr2: gaps below which two fp32 / compensated values may
// be in either true order.  Scratch: this warp's s_ref (double), s_e (int), s_v
// (float), s_l (float), E entries each.  Writes ids[0..k) and wout[0..k).
template <int PL>
__device__ __forceinline__ void select_token(float (&l)[PL], float thr, float thr2, int n_group, int topk_group,
                                             const float* __restrict__ bias, const uint16_t* __restrict__ xrow,
                                             const float* __restrict__ Wg, int H, int E, int k, int renorm,
                                             double* s_ref, int* s_e, float* s_v, float* s_l, int lane,
                                             int32_t* __restrict__ ids, float* __restrict__ wout, WsHeader* hdr) {
    // group-limited top-k: experts of groups that are not kept start out taken
    uint32_t taken = 0;
    if (n_group > 1 && topk_group < n_group) {
        const uint32_t keep = select_groups(l, s_l, s_e, s_ref, E, n_group, topk_group, thr, thr2, xrow, Wg, bias,
                                            H, lane);
        const int gsize = E / n_group;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((keep >> (e / gsize)) & 1u)) taken |= 1u << i;
        }
    }

    // extract candidates in (logit desc, id asc) order until the cluster
    // that contains rank k-1 is closed
    int R = 0;
    float prev_v = 0.f;
    while (R < E) {
        float bv = -INFINITY;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                if (l[i] > bv || (l[i] == bv && e < be)) {
                    bv = l[i];
                    be = e;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be == INT_MAX) break;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == 0) {
            s_e[R] = be;
            s_v[R] = bv;
        }
        ++R;
        if (R >= k + 1) {
            const float gap = prev_v - bv;
            if (!(gap <= thr)) break;
        }
        prev_v = bv;
    }
    __syncwarp();

    // refine each ambiguous cluster that touches ranks 0..k-1
    bool refined = false;
    int a = 0;
    while (a < R && a < k) {
        int b = a;
        while (b + 1 < R && (s_v[b] - s_v[b + 1]) <= thr) ++b;
        if (b > a) {
            refined = true;
            // compensated fp32 values first; fp64 only if they still leave a gap
            // within twice their bound (plus the fp64 rounding of the exact order)
            for (int pass = 0; pass < 2; ++pass) {
                for (int m = a; m <= b; ++m) {
                    const int e = s_e[m];
                    const float* wr = Wg + (int64_t)e * H;
                    double v = pass == 0 ? refine_dot2(xrow, wr, H, lane) : refine_dot(xrow, wr, H, lane);
                    if (bias) v += (double)bias[e];
                    if (lane == 0) s_ref[m] = v;
                }
                __syncwarp();
                if (lane == 0) {  // insertion sort of positions a..b: value desc, id asc
                    for (int m = a + 1; m <= b; ++m) {
                        const double v = s_ref[m];
                        const int e = s_e[m];
                        int q = m - 1;
                        while (q >= a && (s_ref[q] < v || (s_ref[q] == v && s_e[q] > e))) {
                            s_ref[q + 1] = s_ref[q];
                            s_e[q + 1] = s_e[q];
                            --q;
                        }
                        s_ref[q + 1] = v;
                        s_e[q + 1] = e;
                    }
                }
                __syncwarp();
                if (pass == 1) break;
                bool decided = true;
                for (int m = a; m < b; ++m) decided = decided && (s_ref[m] - s_ref[m + 1] > (double)thr2);
                if (decided) break;
            }
            for (int m = a; m <= b; ++m) {  // refined values feed the softmax
                const int e = s_e[m];
                const float v = (float)s_ref[m];
                if ((e & 31) == lane) {
#pragma unroll
                    for (int i = 0; i < PL; ++i)
                        if (i == (e >> 5)) l[i] = v;
                }
            }
        }
        a = b + 1;
    }
    if (refined && lane == 0 && hdr) atomicAdd(&hdr->refined, 1ull);

    // softmax over all E, probabilities of the selected k
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < PL; ++i)
        if (lane + 32 * i < E) mx = fmaxf(mx, l[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i)
        if (lane + 32 * i < E) z += expf(l[i] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);

    float psum = 0.f, my_p = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        const int e = s_e[j];
        const float v = __shfl_sync(0xffffffffu, pick(l, e >> 5), e & 31);
        const float p = expf(v - mx) / z;
        psum += p;
        if (j == lane) {
            my_p = p;
            my_e = e;
        }
    }
    if (lane < k) {
        ids[lane] = my_e;
        wout[lane] = renorm ? my_p / psum : my_p;
    }
    __syncwarp();
}

// max_e ||w_e|| and max_e |b_e| from the split partial squared norms wsq
// [nsplit][E] (block-wide; every thread returns the same values).
__device__ __forceinline__ void weight_norm_max(const float* __restrict__ wsq, int nsplit, int E,
                                                const float* __restrict__ bias, float (*s_red)[32],
                                                float& wnorm_max, float& bias_max) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    float wm = 0.f, bm = 0.f;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float v[RT_MAX_SPLIT];  // all loads in flight before the (ordered) sum
#pragma unroll
        for (int q = 0; q < RT_MAX_SPLIT; ++q) v[q] = q < nsplit ? __ldcg(wsq + (int64_t)q * E + e) : 0.f;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < RT_MAX_SPLIT; ++q) s += v[q];
        wm = fmaxf(wm, s);
        if (bias) bm = fmaxf(bm, fabsf(__ldg(bias + e)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
    }
    if (lane == 0) {
        s_red[0][warp] = wm;
        s_red[1][warp] = bm;
    }
    __syncthreads();
    wm = 0.f;
    bm = 0.f;
    for (int i = 0; i < nw; ++i) {
        wm = fmaxf(wm, s_red[0][i]);
        bm = fmaxf(bm, s_red[1][i]);
    }
    // fp32 bound arithmetic: the threshold coefficients carry a 1 % margin, far above
    // the relative rounding (< 2^-20) of the few fp32 operations on these values
    wnorm_max = sqrtf(wm);
    bias_max = bm;
}

// PL = experts per lane (E <= 32 * PL); lane holds experts lane + 32*i.
template <int PL>
__global__ void __launch_bounds__(RS_WARPS * 32) router_select_kernel(
    const float* __restrict__ part, const float* __restrict__ xsq, const float* __restrict__ wsq, int nsplit,
    float thr_coef, float thr2_coef, int n_group, int topk_group, const float* __restrict__ bias, const uint16_t* __restrict__ x, const float* __restrict__ Wg,
    int64_t T, int H, int E, int k, int renorm, int32_t* __restrict__ ids, float* __restrict__ wout,
    WsHeader* hdr) {
    extern __shared__ __align__(16) unsigned char rs_smem[];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    double* s_ref = reinterpret_cast<double*>(rs_smem) + (size_t)warp * E;
    int* s_e = reinterpret_cast<int*>(reinterpret_cast<double*>(rs_smem) + (size_t)RS_WARPS * E) + (size_t)warp * E;
    float* s_v = reinterpret_cast<float*>(reinterpret_cast<int*>(reinterpret_cast<double*>(rs_smem) +
                                                                 (size_t)RS_WARPS * E) +
                                          (size_t)RS_WARPS * E) +
                 (size_t)warp * E;
    // grouped top-k: this warp's fp32 logits, by expert id
    float* s_l = reinterpret_cast<float*>(rs_smem + (size_t)RS_WARPS * E * (sizeof(double) + sizeof(int) + sizeof(float))) +
                 (size_t)warp * E;
    __shared__ float s_red[2][32];

    // CTA prologue: max_e ||w_e|| and max_e |b_e|
    float wnorm_max, bias_max;
    weight_norm_max(wsq, nsplit, E, bias, s_red, wnorm_max, bias_max);

    for (int64_t t = (int64_t)blockIdx.x * RS_WARPS + warp; t < T; t += (int64_t)gridDim.x * RS_WARPS) {
        // fp32 logits of this token: sum of the split partials in split order, then the bias
        float l[PL];
#pragma unroll
        for (int i = 0; i < PL; ++i) l[i] = 0.f;
        const float* pt = part + t * E + lane;
        constexpr int QB = PL >= 16 ? 1 : 16 / PL;  // splits whose loads are issued together
        for (int q0 = 0; q0 < nsplit; q0 += QB) {
            float v[QB][PL];
#pragma unroll
            for (int b = 0; b < QB; ++b)
#pragma unroll
                for (int i = 0; i < PL; ++i)
                    v[b][i] = (q0 + b < nsplit && lane + 32 * i < E) ? __ldg(pt + (int64_t)(q0 + b) * T * E + 32 * i)
                                                                     : 0.f;
#pragma unroll
            for (int b = 0; b < QB; ++b)
#pragma unroll
                for (int i = 0; i < PL; ++i) l[i] += v[b][i];
        }
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = lane + 32 * i;
            float v = l[i];
            if (e < E) {
                if (bias) v += bias[e];
                if (v != v) v = -INFINITY;  // NaN logits never win
            } else {
                v = -INFINITY;
            }
            l[i] = v;
        }
        // squared norm of x_t: only bounds the error (inflated by 1.01), order is immaterial
        float xs2 = 0.f;
        for (int q = lane; q < nsplit; q += 32) xs2 += xsq[(int64_t)q * T + t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) xs2 += __shfl_xor_sync(0xffffffffu, xs2, off);
        // two fp32 logits closer than thr may be in either true order
        const float thr = thr_coef * fmaf(sqrtf(xs2), wnorm_max, bias_max);
        // the same for the compensated values (twice their bound)
        const float thr2 = thr2_coef * fmaf(sqrtf(xs2), wnorm_max, bias_max);
        select_token<PL>(l, thr, thr2, n_group, topk_group, bias, x + t * (int64_t)H, Wg, H, E, k, renorm, s_ref,
                         s_e, s_v, s_l, lane, ids + t * k, wout + t * k, hdr);
    }
}

// ---------------------------------------------------------------------------
// Small batches (decode): one launch for logits and selection.
//
// Each CTA (16 warps) stages the T <= 16 token rows in shared memory, then
// computes the complete logits of `epb` experts: warp w takes expert
// epb * blockIdx.x + (w % epb) over part (w / epb) of the QN = 16 / epb parts of
// H.  Lane l of a part takes its 8-element pieces l, l + 32, ...; piece i of a
// lane feeds accumulator (i & 1) of each token with 8 chained fmas; the two
// accumulators are added, the lanes summed by an xor butterfly, and the parts in
// part order, so a logit's rounding depth is n = 8 ceil(npl / 2) + 1 + 5 +
// (QN - 1) (+ 1 for the bias), npl = pieces per lane.  The squared row norms of
// Wg come out of the same loads.  The logits and norms go to the workspace; the
// CTA that finishes last (a ticket in the workspace header) runs the selection
// of every token -- one warp per token, as router_select_kernel does -- with the
// bound of this depth.  Non-last CTAs simply exit; the last one puts the ticket
// back to 0 before it lets the next kernel launch, so launches never overlap
// on the ticket.
constexpr int RSM_WARPS = 16;
constexpr int RSM_THREADS = RSM_WARPS * 32;
constexpr int RSM_MAX_T = 16;
constexpr int RSM_MAX_NPL = 8;  // pieces per lane: all of a lane's weight loads in flight at once

template <int PL>
__global__ void __launch_bounds__(RSM_THREADS, 1) router_small_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ Wg, const float* __restrict__ bias, int T, int H,
    int E, int k, int renorm, int epb, float thr_coef, float thr2_coef, int n_group, int topk_group,
    float* __restrict__ lg, float* __restrict__ wsq, int32_t* __restrict__ ids, float* __restrict__ wout,
    WsHeader* hdr) {
    extern __shared__ __align__(16) unsigned char rsm[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(rsm);                              // [T][H]
    float* part = reinterpret_cast<float*>(rsm + (size_t)T * H * 2);             // [RSM_WARPS][T]
    float* wpart = part + RSM_WARPS * RSM_MAX_T;                                 // [RSM_WARPS]
    unsigned char* sel = reinterpret_cast<unsigned char*>(wpart + RSM_WARPS);   // select scratch
    __shared__ float s_red[2][32];
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();

    // token rows -> shared memory (one round trip for all of them)
    const int nvec = T * H / 8;
    for (int i = tid; i < nvec; i += RSM_THREADS) cp_async16(xs + (size_t)i * 8, x + (size_t)i * 8, true);
    cp_async_commit();

    const int QN = RSM_WARPS / epb;
    const int jw = warp % epb, q = warp / epb;
    const int e = blockIdx.x * epb + jw;
    const int NP = H / 8;
    const int pb = (int)((int64_t)NP * q / QN), pe = (int)((int64_t)NP * (q + 1) / QN);
    // this lane's weight pieces, all loads issued before the first use
    float4 wv[RSM_MAX_NPL][2];
    const float* wrow = Wg + (int64_t)(e < E ? e : 0) * H;
#pragma unroll
    for (int i = 0; i < RSM_MAX_NPL; ++i) {
        const int pc = pb + lane + 32 * i;
        const bool ok = e < E && pc < pe;
        wv[i][0] = ok ? __ldg(reinterpret_cast<const float4*>(wrow) + 2 * pc) : make_float4(0.f, 0.f, 0.f, 0.f);
        wv[i][1] = ok ? __ldg(reinterpret_cast<const float4*>(wrow) + 2 * pc + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float wn = 0.f;
#pragma unroll
    for (int i = 0; i < RSM_MAX_NPL; ++i) {
        wn = fmaf(wv[i][0].x, wv[i][0].x, wn); wn = fmaf(wv[i][0].y, wv[i][0].y, wn);
        wn = fmaf(wv[i][0].z, wv[i][0].z, wn); wn = fmaf(wv[i][0].w, wv[i][0].w, wn);
        wn = fmaf(wv[i][1].x, wv[i][1].x, wn); wn = fmaf(wv[i][1].y, wv[i][1].y, wn);
        wn = fmaf(wv[i][1].z, wv[i][1].z, wn); wn = fmaf(wv[i][1].w, wv[i][1].w, wn);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wn += __shfl_xor_sync(0xffffffffu, wn, off);
    cp_async_wait_group<0>();
    __syncthreads();

    for (int t = 0; t < T; ++t) {
        const uint16_t* xr = xs + (size_t)t * H;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < RSM_MAX_NPL; ++i) {
            const int pc = pb + lane + 32 * i;
            if (pc < pe) {
                float xf[8];
                unpack8(*reinterpret_cast<const uint4*>(xr + (size_t)pc * 8), xf);
                float a = (i & 1) ? a1 : a0;
                a = fmaf(xf[0], wv[i][0].x, a); a = fmaf(xf[1], wv[i][0].y, a);
                a = fmaf(xf[2], wv[i][0].z, a); a = fmaf(xf[3], wv[i][0].w, a);
                a = fmaf(xf[4], wv[i][1].x, a); a = fmaf(xf[5], wv[i][1].y, a);
                a = fmaf(xf[6], wv[i][1].z, a); a = fmaf(xf[7], wv[i][1].w, a);
                if (i & 1) a1 = a; else a0 = a;
            }
        }
        float v = a0 + a1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) part[warp * RSM_MAX_T + t] = v;
    }
    if (lane == 0) wpart[warp] = wn;
    __syncthreads();
    // the parts of each logit in part order (warp jw + epb * q holds part q of expert jw)
    for (int i = tid; i < epb * T; i += RSM_THREADS) {
        const int jj = i % epb, t = i / epb, ee = blockIdx.x * epb + jj;
        if (ee >= E) continue;
        float v = part[jj * RSM_MAX_T + t];
        for (int qq = 1; qq < QN; ++qq) v += part[(jj + epb * qq) * RSM_MAX_T + t];
        lg[(int64_t)t * E + ee] = v;
    }
    if (tid < epb && blockIdx.x * epb + tid < E) {
        float v = wpart[tid];
        for (int qq = 1; qq < QN; ++qq) v += wpart[tid + epb * qq];
        wsq[blockIdx.x * epb + tid] = v;
    }
    // publish, then take a ticket; the last CTA to arrive sees every CTA's writes
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&hdr->route_ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    if (tid == 0) hdr->route_ticket = 0u;  // every CTA of this launch has taken its ticket
    __threadfence();
    pdl_trigger();

    // ---- selection, one warp per token (the last CTA only) ----
    float wnorm_max, bias_max;
    weight_norm_max(wsq, 1, E, bias, s_red, wnorm_max, bias_max);
    double* s_ref = reinterpret_cast<double*>(sel) + (size_t)warp * E;
    int* s_e = reinterpret_cast<int*>(reinterpret_cast<double*>(sel) + (size_t)RSM_WARPS * E) + (size_t)warp * E;
    float* s_v = reinterpret_cast<float*>(reinterpret_cast<int*>(reinterpret_cast<double*>(sel) +
                                                                 (size_t)RSM_WARPS * E) +
                                          (size_t)RSM_WARPS * E) +
                 (size_t)warp * E;
    float* s_l = reinterpret_cast<float*>(sel + (size_t)RSM_WARPS * E * (sizeof(double) + sizeof(int) + sizeof(float))) +
                 (size_t)warp * E;
    if (warp >= T) return;
    const int t = warp;
    float l[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int ee = lane + 32 * i;
        float v = -INFINITY;
        if (ee < E) {
            v = __ldcg(lg + (int64_t)t * E + ee);
            if (bias) v += bias[ee];
            if (v != v) v = -INFINITY;  // NaN logits never win
        }
        l[i] = v;
    }
    // squared norm of x_t: only bounds the error (inflated by 1.01), order is immaterial
    float xs2 = 0.f;
    for (int pc = lane; pc < NP; pc += 32) {
        float xf[8];
        unpack8(*reinterpret_cast<const uint4*>(xs + (size_t)t * H + (size_t)pc * 8), xf);
#pragma unroll
        for (int i = 0; i < 8; ++i) xs2 = fmaf(xf[i], xf[i], xs2);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) xs2 += __shfl_xor_sync(0xffffffffu, xs2, off);
    const float thr = thr_coef * fmaf(sqrtf(xs2), wnorm_max, bias_max);
    const float thr2 = thr2_coef * fmaf(sqrtf(xs2), wnorm_max, bias_max);
    select_token<PL>(l, thr, thr2, n_group, topk_group, bias, x + (int64_t)t * H, Wg, H, E, k, renorm, s_ref, s_e,
                     s_v, s_l, lane, ids + (int64_t)t * k, wout + (int64_t)t * k, hdr);
}

}  // namespace

// Split of H into K ranges: the CTAs run in waves of two CTAs per SM, so pick the
// range length that minimises waves x (range + a fixed per-CTA overhead of about
// three chunks).
void router_plan(int64_t T, int H, int E, int num_sms, int* nsplit, int* KC) {
    const int64_t tT = (T + RT_BT - 1) / RT_BT;
    const int64_t tE = (E + RT_BE - 1) / RT_BE;
    const int64_t base = tT * tE;
    const int64_t slots = std::max<int64_t>(1, std::min<int64_t>(2 * (int64_t)num_sms, RT_TARGET_MAX));
    int best_kc = H, best_ns = 1;
    int64_t best_cost = INT64_MAX;
    for (int kc = RT_BK; kc <= H; kc += RT_BK) {
        const int ns = (H + kc - 1) / kc;
        if (ns > RT_MAX_SPLIT) continue;
        if ((int64_t)(ns - 1) * kc >= H) continue;  // same split as a shorter range
        if (base * ns > RT_TARGET_MAX + base) continue;  // the workspace is sized for this bound
        const int64_t waves = (base * ns + slots - 1) / slots;
        const int64_t cost = waves * (kc + 3 * RT_BK);
        if (cost < best_cost) {
            best_cost = cost;
            best_kc = kc;
            best_ns = ns;
        }
    }
    *KC = best_kc;
    *nsplit = best_ns;
}

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Scratch of the router for up to T tokens, for any split plan router_plan can
// choose: nsplit * ceil(T/128) * ceil(E/64) < RT_TARGET_MAX + ceil(T/128) * ceil(E/64).
static void router_sizes(int64_t T, int E, size_t* part, size_t* xs, size_t* ws) {
    const int64_t tT = (T + RT_BT - 1) / RT_BT;
    const int64_t tE = (E + RT_BE - 1) / RT_BE;
    *part = align256((size_t)(RT_TARGET_MAX + tT * tE) * RT_BT * RT_BE * sizeof(float));
    *xs = align256((size_t)RT_MAX_SPLIT * (size_t)T * sizeof(float));
    *ws = align256((size_t)RT_MAX_SPLIT * (size_t)E * sizeof(float));
}

size_t router_scratch_bytes(int64_t T, int H, int E, int num_sms) {
    (void)num_sms;
    (void)H;
    size_t a, b, c;
    router_sizes(T, E, &a, &b, &c);
    return a + b + c;
}

void router_carve(void* base, int64_t T, int E, float** part, float** xsq, float** wsq) {
    size_t a, b, c;
    router_sizes(T, E, &a, &b, &c);
    char* p = static_cast<char*>(base);
    *part = reinterpret_cast<float*>(p);
    *xsq = reinterpret_cast<float*>(p + a);
    *wsq = reinterpret_cast<float*>(p + a + b);
}

// Plan of the small-batch router: experts per CTA (epb) and parts of H per
// expert (16 / epb), or false if the batch does not fit its envelope.
static bool small_router_plan(const RouterLaunch& L, int* epb, size_t* smem) {
    if (!L.hdr || L.T < 1 || L.T > RSM_MAX_T) return false;
    const int NP = L.H / 8;
    int qn_min = 1;
    while (qn_min < RSM_WARPS && (NP + qn_min - 1) / qn_min > 32 * RSM_MAX_NPL) qn_min <<= 1;
    if ((NP + qn_min - 1) / qn_min > 32 * RSM_MAX_NPL) return false;
    int e = 1;
    while (e * 2 <= RSM_WARPS / qn_min && e * 2 * 16 <= L.E) e <<= 1;
    *epb = e;
    *smem = (size_t)L.T * L.H * 2 + sizeof(float) * (RSM_WARPS * RSM_MAX_T + RSM_WARPS) +
            (size_t)RSM_WARPS * L.E * (sizeof(double) + sizeof(int) + 2 * sizeof(float));
    return *smem <= 200 * 1024;
}

cudaError_t launch_router(const RouterLaunch& L, int num_sms, cudaStream_t s) {
    const double u32 = 1.0 / 16777216.0, u64 = 1.0 / 9007199254740992.0;
    const double g64 = (L.H + 2.0) * u64 / (1.0 - (L.H + 2.0) * u64);
    // compensated recheck: (gamma_{ceil(H/128)} + gamma_128)^2 per value, plus
    // the fp64 rounding of the exact order and of hi + lo + bias
    const double na = (L.H + 127) / 128, nc = 128.0;
    const double ga = na * u32 / (1.0 - na * u32), gc = nc * u32 / (1.0 - nc * u32);
    const float thr2_coef = (float)(2.0 * ((ga + gc) * (ga + gc) + g64 + 3.0 * u64) * 1.01);

    int epb = 1;
    size_t smem_small = 0;
    if (small_router_plan(L, &epb, &smem_small)) {
        // rounding depth of the small kernel: the fma chains of one accumulator (8 per
        // piece), the two accumulators, the lane butterfly, the parts of H, the bias
        const int QN = RSM_WARPS / epb;
        const int NP = L.H / 8;
        const int npl = ((NP + QN - 1) / QN + 31) / 32;
        const int chain_n = 8 * ((npl + 1) / 2) + 1 + 5 + (QN - 1) + 1;
        const double g32 = chain_n * u32 / (1.0 - chain_n * u32);
        const float thr_coef = (float)(2.0 * (g32 + g64) * 1.01);
        const unsigned grid = (unsigned)((L.E + epb - 1) / epb);
        cudaError_t err = cudaSuccess;
#define MOE_SMALL(PLV)                                                                                           \
    do {                                                                                                         \
        err = cudaFuncSetAttribute(router_small_kernel<PLV>, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                   (int)smem_small);                                                             \
        if (err != cudaSuccess) return err;                                                                      \
        err = launch_k("router_small", router_small_kernel<PLV>, dim3(grid), dim3(RSM_THREADS), smem_small, s,   \
                       L.x, L.Wg, L.bias, (int)L.T, L.H, L.E, L.k, L.renorm, epb, thr_coef, thr2_coef, L.n_group, \
                       L.topk_group, L.part, L.wsq, L.ids, L.w, L.hdr);                                          \
    } while (0)
        if (L.E <= 32)
            MOE_SMALL(1);
        else if (L.E <= 64)
            MOE_SMALL(2);
        else if (L.E <= 128)
            MOE_SMALL(4);
        else if (L.E <= 256)
            MOE_SMALL(8);
        else
            MOE_SMALL(16);
#undef MOE_SMALL
        return err;
    }

    const int64_t tT = (L.T + RT_BT - 1) / RT_BT;
    const int tE = (L.E + RT_BE - 1) / RT_BE;
    dim3 grid1((unsigned)tE, (unsigned)tT, (unsigned)L.nsplit);
    cudaError_t err = cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)RT_SMEM);
    if (err != cudaSuccess) return err;
    err = launch_k("router_logits", router_logits_kernel, grid1, dim3(RT_THREADS), RT_SMEM, s, L.x, L.Wg, L.T, L.H,
                   L.E, L.KC, L.part, L.xsq, L.wsq);
    if (err != cudaSuccess) return err;

    // worst-case rounding depth of one logit: 32-term chunk, 8-chunk group,
    // groups in the CTA range, split partials, bias
    const int groups = (L.KC + RT_BK * RT_GROUP - 1) / (RT_BK * RT_GROUP);
    // rounding depth: the 32-term chain of a chunk, 8 chunks of a group, the groups
    // of the range, the split partials, the bias
    const int chain_n = RT_BK + RT_GROUP + groups + L.nsplit + 1;
    // per-logit bound B_t = (gamma_n(fp32) + gamma_{H+2}(fp64)) * (||x_t|| max||w_e|| + max|b_e|);
    // threshold on a gap = 2 B_t, with a 1 % margin that covers the fp32 evaluation
    const double g32 = chain_n * u32 / (1.0 - chain_n * u32);
    const float thr_coef = (float)(2.0 * (g32 + g64) * 1.01);
    const size_t smem = (size_t)RS_WARPS * L.E * (sizeof(double) + sizeof(int) + 2 * sizeof(float));
    const int64_t want = (L.T + RS_WARPS - 1) / RS_WARPS;
    const unsigned grid2 = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
#define MOE_SELECT(PLV)                                                                                          \
    do {                                                                                                         \
        if (smem > 48 * 1024) {                                                                                  \
            err = cudaFuncSetAttribute(router_select_kernel<PLV>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                                       (int)smem);                                                               \
            if (err != cudaSuccess) return err;                                                                  \
        }                                                                                                        \
        err = launch_k("router_select", router_select_kernel<PLV>, dim3(grid2), dim3(RS_WARPS * 32), smem, s,    \
                       L.part, L.xsq, L.wsq, L.nsplit, thr_coef, thr2_coef, L.n_group, L.topk_group, L.bias, L.x,   \
                       L.Wg, L.T, L.H, L.E, L.k, L.renorm, L.ids, L.w, L.hdr);                                   \
    } while (0)
    if (L.E <= 32)
        MOE_SELECT(1);
    else if (L.E <= 64)
        MOE_SELECT(2);
    else if (L.E <= 128)
        MOE_SELECT(4);
    else if (L.E <= 256)
        MOE_SELECT(8);
    else
        MOE_SELECT(16);
#undef MOE_SELECT
    return err;
}

}  // namespace moe
