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
//     Tile 64 tokens x 64 experts x K-range; each thread owns 4x4 outputs.
//     Accumulation is nested (32-term chunks -> groups of 8 chunks -> the
//     CTA's range), which keeps the worst-case rounding error of every logit
//     below gamma_n * (||x_t|| ||w_e|| + |b_e|) with a small n (about 70 for
//     H = 7168) instead of n = H.  The CTAs of the first token/expert tile
//     also emit the partial squared norms of x rows and Wg rows.
//  2. router_select_kernel: one warp per token.  Sums the split partials in
//     fixed order, adds the bias, and takes the k+1 largest logits (ties ->
//     lower id).  Consecutive candidates whose fp32 gap is within twice the
//     per-token bound form a cluster whose true order fp32 cannot decide; each
//     cluster that touches the top k is recomputed in fp64 from the exact
//     bf16 x fp32 products and re-ordered (ties -> lower id).  Then the fp32
//     softmax (expf) over all E logits, the selected probabilities, and the
//     optional renormalisation (divide by their sum, in j order).
#include <float.h>
#include <limits.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int RT_BT = 64;        // tokens per CTA
constexpr int RT_BE = 64;        // experts per CTA
constexpr int RT_BK = 32;        // K per shared-memory chunk (level-1 sum length)
constexpr int RT_GROUP = 8;      // chunks per level-2 group
constexpr int RT_THREADS = 256;
constexpr int RT_TARGET_MAX = 2048;  // upper bound on CTAs the split plan aims for
constexpr int RT_MAX_SPLIT = 32;

constexpr int RS_WARPS = 8;      // select: tokens (warps) per CTA
constexpr int RS_MAXE = 512;
constexpr int RS_PER_LANE = RS_MAXE / 32;

__global__ void __launch_bounds__(RT_THREADS) router_logits_kernel(const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ Wg, int64_t T,
                                                                   int H, int E, int KC,
                                                                   float* __restrict__ part,
                                                                   float* __restrict__ xsq,
                                                                   float* __restrict__ wsq) {
    __shared__ __align__(16) float xs[2][RT_BK][RT_BT + 4];
    __shared__ __align__(16) float wsm[2][RT_BK][RT_BE + 4];

    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * RT_BT;
    const int e0 = blockIdx.y * RT_BE;
    const int sp = blockIdx.z;
    const int kbeg = sp * KC;
    const int kend = min(H, kbeg + KC);
    const int nchunk = (kend - kbeg) / RT_BK;

    // loader: thread -> (row of the tile, 8 consecutive k)
    const int lrow = tid >> 2;
    const int lk = (tid & 3) * 8;
    const int64_t xt = t0 + lrow;
    const bool xvalid = xt < T;
    const int we = e0 + lrow;
    const bool wvalid = we < E;
    const uint16_t* xsrc = x + (xvalid ? xt : 0) * (int64_t)H + kbeg + lk;
    const float* wsrc = Wg + (int64_t)(wvalid ? we : 0) * H + kbeg + lk;

    uint4 xr = make_uint4(0, 0, 0, 0);
    float4 wr0 = make_float4(0.f, 0.f, 0.f, 0.f), wr1 = wr0;
    auto gload = [&](int c) {
        if (xvalid) xr = __ldg(reinterpret_cast<const uint4*>(xsrc + c * RT_BK));
        if (wvalid) {
            wr0 = __ldg(reinterpret_cast<const float4*>(wsrc + c * RT_BK));
            wr1 = __ldg(reinterpret_cast<const float4*>(wsrc + c * RT_BK + 4));
        }
    };
    auto sstore = [&](int buf) {
        float f[8];
        unpack8(xr, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) xs[buf][lk + i][lrow] = f[i];
        wsm[buf][lk + 0][lrow] = wr0.x;
        wsm[buf][lk + 1][lrow] = wr0.y;
        wsm[buf][lk + 2][lrow] = wr0.z;
        wsm[buf][lk + 3][lrow] = wr0.w;
        wsm[buf][lk + 4][lrow] = wr1.x;
        wsm[buf][lk + 5][lrow] = wr1.y;
        wsm[buf][lk + 6][lrow] = wr1.z;
        wsm[buf][lk + 7][lrow] = wr1.w;
    };

    const int ty = tid >> 4;  // tokens ty*4 .. +3
    const int tx = tid & 15;  // experts tx*4 .. +3
    const bool do_xn = (blockIdx.y == 0) && (tid < RT_BT);
    const bool do_wn = (blockIdx.x == 0) && (tid >= 64) && (tid < 64 + RT_BE);
    float a1[4][4], a2[4][4], a3[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a1[i][j] = a2[i][j] = a3[i][j] = 0.f;
    float nsq = 0.f;

    if (nchunk > 0) {
        gload(0);
        sstore(0);
    }
    __syncthreads();
    for (int c = 0; c < nchunk; ++c) {
        const int buf = c & 1;
        if (c + 1 < nchunk) gload(c + 1);
#pragma unroll 8
        for (int kk = 0; kk < RT_BK; ++kk) {
            const float4 av = *reinterpret_cast<const float4*>(&xs[buf][kk][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4*>(&wsm[buf][kk][tx * 4]);
            const float a[4] = {av.x, av.y, av.z, av.w};
            const float b[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) a1[i][j] = fmaf(a[i], b[j], a1[i][j]);
        }
        if (do_xn) {
#pragma unroll 8
            for (int kk = 0; kk < RT_BK; ++kk) {
                const float v = xs[buf][kk][tid];
                nsq = fmaf(v, v, nsq);
            }
        } else if (do_wn) {
#pragma unroll 8
            for (int kk = 0; kk < RT_BK; ++kk) {
                const float v = wsm[buf][kk][tid - 64];
                nsq = fmaf(v, v, nsq);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a2[i][j] += a1[i][j];
                a1[i][j] = 0.f;
            }
        if ((c % RT_GROUP) == RT_GROUP - 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    a3[i][j] += a2[i][j];
                    a2[i][j] = 0.f;
                }
        }
        if (c + 1 < nchunk) sstore(buf ^ 1);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a3[i][j] += a2[i][j];

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + ty * 4 + i;
        if (t >= T) continue;
        float* dst = part + ((int64_t)sp * T + t) * E;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) dst[e] = a3[i][j];
        }
    }
    if (do_xn && t0 + tid < T) xsq[(int64_t)sp * T + t0 + tid] = nsq;
    if (do_wn && e0 + (tid - 64) < E) wsq[(int64_t)sp * E + e0 + (tid - 64)] = nsq;
}

// fp64 dot product of one bf16 x row with one fp32 Wg row, by one warp.
// Every lane returns the same value (xor-butterfly sums are symmetric).
__device__ double refine_dot(const uint16_t* __restrict__ xrow, const float* __restrict__ wrow, int H, int lane) {
    double s = 0.0;
    for (int h0 = lane * 8; h0 < H; h0 += 256) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xrow + h0));
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(wrow + h0));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(wrow + h0 + 4));
        float xf[8];
        unpack8(xv, xf);
        s = fma((double)xf[0], (double)w0.x, s);
        s = fma((double)xf[1], (double)w0.y, s);
        s = fma((double)xf[2], (double)w0.z, s);
        s = fma((double)xf[3], (double)w0.w, s);
        s = fma((double)xf[4], (double)w1.x, s);
        s = fma((double)xf[5], (double)w1.y, s);
        s = fma((double)xf[6], (double)w1.z, s);
        s = fma((double)xf[7], (double)w1.w, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

__device__ __forceinline__ double gamma_n(double n, double u) { return n * u / (1.0 - n * u); }

__device__ __forceinline__ float pick(const float (&l)[RS_PER_LANE], int idx) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < RS_PER_LANE; ++i)
        if (i == idx) v = l[i];
    return v;
}

__global__ void __launch_bounds__(RS_WARPS * 32) router_select_kernel(
    const float* __restrict__ part, const float* __restrict__ xsq, const float* __restrict__ wsq, int nsplit,
    int chain_n, const float* __restrict__ bias, const uint16_t* __restrict__ x, const float* __restrict__ Wg,
    int64_t T, int H, int E, int k, int renorm, int32_t* __restrict__ ids, float* __restrict__ wout,
    WsHeader* hdr) {
    extern __shared__ __align__(16) unsigned char rs_smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    double* s_ref = reinterpret_cast<double*>(rs_smem) + (size_t)warp * E;
    int* s_e = reinterpret_cast<int*>(reinterpret_cast<double*>(rs_smem) + (size_t)RS_WARPS * E) + (size_t)warp * E;
    float* s_v = reinterpret_cast<float*>(reinterpret_cast<int*>(reinterpret_cast<double*>(rs_smem) +
                                                                 (size_t)RS_WARPS * E) +
                                          (size_t)RS_WARPS * E) +
                 (size_t)warp * E;
    __shared__ float s_red[2][RS_WARPS];

    // CTA prologue: max_e ||w_e||^2 and max_e |b_e|
    float wm = 0.f, bm = 0.f;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < nsplit; ++q) s += wsq[(int64_t)q * E + e];
        wm = fmaxf(wm, s);
        if (bias) bm = fmaxf(bm, fabsf(bias[e]));
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
    for (int i = 0; i < RS_WARPS; ++i) {
        wm = fmaxf(wm, s_red[0][i]);
        bm = fmaxf(bm, s_red[1][i]);
    }
    const double wnorm_max = sqrt((double)wm);
    const double bias_max = (double)bm;
    const double g32 = gamma_n((double)chain_n, 1.0 / 16777216.0);             // u = 2^-24
    const double g64 = gamma_n((double)H + 2.0, 1.0 / 9007199254740992.0);      // u = 2^-53

    for (int64_t t = (int64_t)blockIdx.x * RS_WARPS + warp; t < T; t += (int64_t)gridDim.x * RS_WARPS) {
        // fp32 logits of this token: lane holds experts lane + 32*i
        float l[RS_PER_LANE];
#pragma unroll
        for (int i = 0; i < RS_PER_LANE; ++i) {
            const int e = lane + 32 * i;
            float v = -INFINITY;
            if (e < E) {
                v = 0.f;
                for (int q = 0; q < nsplit; ++q) v += part[((int64_t)q * T + t) * E + e];
                if (bias) v += bias[e];
                if (v != v) v = -INFINITY;  // NaN logits never win
            }
            l[i] = v;
        }
        float xs2 = 0.f;
        for (int q = 0; q < nsplit; ++q) xs2 += xsq[(int64_t)q * T + t];
        const double mag = (sqrt((double)xs2) * wnorm_max + bias_max) * 1.01;
        const double thr = 2.0 * (g32 + g64) * mag;  // two logits closer than this: order not certain

        // extract candidates in (logit desc, id asc) order until the cluster
        // that contains rank k-1 is closed
        uint32_t taken = 0;
        int R = 0;
        float prev_v = 0.f;
        while (R < E) {
            float bv = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < RS_PER_LANE; ++i) {
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
                const double gap = (double)prev_v - (double)bv;
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
            while (b + 1 < R && ((double)s_v[b] - (double)s_v[b + 1]) <= thr) ++b;
            if (b > a) {
                refined = true;
                for (int m = a; m <= b; ++m) {
                    const int e = s_e[m];
                    double v = refine_dot(x + t * (int64_t)H, Wg + (int64_t)e * H, H, lane);
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
                for (int m = a; m <= b; ++m) {  // refined values feed the softmax
                    const int e = s_e[m];
                    const float v = (float)s_ref[m];
                    if ((e & 31) == lane) {
#pragma unroll
                        for (int i = 0; i < RS_PER_LANE; ++i)
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
        for (int i = 0; i < RS_PER_LANE; ++i)
            if (lane + 32 * i < E) mx = fmaxf(mx, l[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < RS_PER_LANE; ++i)
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
            ids[t * k + lane] = my_e;
            wout[t * k + lane] = renorm ? my_p / psum : my_p;
        }
        __syncwarp();
    }
}

}  // namespace

void router_plan(int64_t T, int H, int E, int num_sms, int* nsplit, int* KC) {
    const int64_t tT = (T + RT_BT - 1) / RT_BT;
    const int64_t tE = (E + RT_BE - 1) / RT_BE;
    const int64_t base = tT * tE;
    const int64_t target = std::min<int64_t>(2 * (int64_t)num_sms, RT_TARGET_MAX);
    int64_t ns = (target + base - 1) / base;
    const int64_t ns_max = std::max(1, std::min(RT_MAX_SPLIT, H / 256));
    ns = std::max<int64_t>(1, std::min(ns, ns_max));
    int kc = (int)((H + ns - 1) / ns);
    kc = (kc + RT_BK - 1) / RT_BK * RT_BK;
    *KC = kc;
    *nsplit = (H + kc - 1) / kc;
}

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Scratch of the router for up to T tokens, for any split plan router_plan can
// choose: nsplit * ceil(T/64) * ceil(E/64) < RT_TARGET_MAX + ceil(T/64) * ceil(E/64).
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

cudaError_t launch_router(const RouterLaunch& L, int num_sms, cudaStream_t s) {
    const int64_t tT = (L.T + RT_BT - 1) / RT_BT;
    const int tE = (L.E + RT_BE - 1) / RT_BE;
    dim3 grid1((unsigned)tT, (unsigned)tE, (unsigned)L.nsplit);
    router_logits_kernel<<<grid1, RT_THREADS, 0, s>>>(L.x, L.Wg, L.T, L.H, L.E, L.KC, L.part, L.xsq, L.wsq);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    // worst-case rounding depth of one logit: 32-term chunk, 8-chunk group,
    // groups in the CTA range, split partials, bias
    const int groups = (L.KC + RT_BK * RT_GROUP - 1) / (RT_BK * RT_GROUP);
    const int chain_n = RT_BK + RT_GROUP + groups + L.nsplit + 1;
    const size_t smem = (size_t)RS_WARPS * L.E * (sizeof(double) + sizeof(int) + sizeof(float));
    if (smem > 48 * 1024) {
        err = cudaFuncSetAttribute(router_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    const int64_t want = (L.T + RS_WARPS - 1) / RS_WARPS;
    const unsigned grid2 = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
    router_select_kernel<<<grid2, RS_WARPS * 32, smem, s>>>(L.part, L.xsq, L.wsq, L.nsplit, chain_n, L.bias, L.x,
                                                             L.Wg, L.T, L.H, L.E, L.k, L.renorm, L.ids, L.w, L.hdr);
    return cudaGetLastError();
}

}  // namespace moe
