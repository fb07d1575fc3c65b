// moe_api.cu -- the C ABI of include/moe.h: argument checks, workspace
// carve-up and kernel launches.  No allocation, no host synchronisation
// (except the two explicit status readers).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "moe_internal.cuh"

using namespace moe;

namespace {

std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<int> g_pair_mode{0};
std::atomic<int> g_pdl{1};
std::atomic<uint64_t> g_launches{0};

// Launch-event hook (moe_launch_events_arm): the caller's events, how many are
// used, and the label of each used one.
struct LaunchEvents {
    std::mutex mu;
    std::vector<cudaEvent_t> events;
    std::vector<std::string> labels;
};
LaunchEvents g_ev;
std::atomic<int> g_ev_armed{0};

// Records the next armed event on s (an external node under stream capture).
cudaError_t record_next_event(const char* label, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_ev.mu);
    if (g_ev.labels.size() >= g_ev.events.size()) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    e = cudaEventRecordWithFlags(g_ev.events[g_ev.labels.size()], s,
                                 cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
    if (e != cudaSuccess) return e;
    g_ev.labels.emplace_back(label);
    return cudaSuccess;
}

int device_sms() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

size_t a256(size_t v) { return (v + 255) & ~(size_t)255; }

// Small batches split the shared expert's FC2 into K ranges of about the routed
// FC2's length, so its tiles do not outlast the routed ones; the fp32 partials
// are summed by the combine.
constexpr int64_t kSplitMaxT = 128;
constexpr int kSplitMax = 8;

int shared_split(int64_t T, int I, int I_sh) {
    if (I_sh <= 0 || T <= 0 || T > kSplitMaxT) return 1;
    const int r = I_sh / I;
    return r < 2 ? 1 : (r > kSplitMax ? kSplitMax : r);
}

struct ForwardLayout {
    size_t h, h_sh, y, y_sh, y_sh_part;
    // E4M3 activations: quantised expert inputs, shared input, intermediates, and scales
    // (NVFP4 activations keep their packed codes and row scales in the same regions)
    size_t xq, sxq, xsq, sxs, hq, shq, hsq, shs;
    // NVFP4 activations: block scales of the expert inputs, shared input, intermediates
    size_t xsf, xssf, hsf, hssf;
    size_t total;
};

ForwardLayout forward_layout(int64_t P_cap, int64_t T, int H, int I, int I_sh) {
    ForwardLayout L;
    size_t off = kWsHeaderBytes;
    L.h = off;
    off += a256((size_t)P_cap * (size_t)I * 2);
    L.h_sh = off;
    off += a256((size_t)(I_sh > 0 ? T : 0) * (size_t)I_sh * 2);
    L.y = off;
    off += a256((size_t)P_cap * (size_t)H * 2);
    L.y_sh = off;
    off += a256((size_t)(I_sh > 0 ? T : 0) * (size_t)H * 2);
    L.y_sh_part = off;
    const int ks = shared_split(T, I, I_sh);
    off += a256(ks > 1 ? (size_t)ks * (size_t)T * (size_t)H * 4 : 0);
    const size_t T_sh = I_sh > 0 ? (size_t)T : 0;
    L.xq = off;
    off += a256((size_t)P_cap * (size_t)H);
    L.sxq = off;
    off += a256((size_t)P_cap * 4);
    L.xsq = off;
    off += a256(T_sh * (size_t)H);
    L.sxs = off;
    off += a256(T_sh * 4);
    L.hq = off;
    off += a256((size_t)P_cap * (size_t)I);
    L.shq = off;
    off += a256((size_t)P_cap * 4);
    L.hsq = off;
    off += a256(T_sh * (size_t)(I_sh > 0 ? I_sh : 0));
    L.shs = off;
    off += a256(T_sh * 4);
    L.xsf = off;
    off += a256((size_t)P_cap * (size_t)nvfp4_sf_row_bytes(H));
    L.xssf = off;
    off += a256(T_sh * (size_t)nvfp4_sf_row_bytes(H));
    L.hsf = off;
    off += a256((size_t)P_cap * (size_t)nvfp4_sf_row_bytes(I));
    L.hssf = off;
    off += a256(T_sh * (size_t)(I_sh > 0 ? nvfp4_sf_row_bytes(I_sh) : 0));
    L.total = off;
    return L;
}

size_t route_need(int64_t T, int H, int E) { return kWsHeaderBytes + router_scratch_bytes(T, H, E, 0); }
size_t permute_need(int64_t P, int S_local) { return kWsHeaderBytes + permute_scratch_bytes(P, S_local); }

bool dim_ok(int v) { return v > 0 && v % 64 == 0 && v <= (1 << 20); }

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

// An NVTX range around each entry point of the ABI (a profiler's timeline shows
// which call enqueued which kernels; without a tool attached it costs a check).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define MOE_NVTX(name) NvtxRange moe_nvtx_range_(name)

bool moe::pdl_enabled() { return g_pdl.load() != 0 && g_ev_armed.load() == 0; }

cudaError_t moe::note_launch(const char* name, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return g_ev_armed.load() ? record_next_event(name, s) : cudaSuccess;
}

extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported size";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_BOUNDS: return "device: id out of range";
        case MOE_ERR_TIMEOUT: return "device: bounded wait timed out";
        case MOE_ERR_DEVICE_BOUNDS | MOE_ERR_TIMEOUT: return "device: id out of range and wait timed out";
        default: return "unknown status";
    }
}

void moe_set_wait_timeout_ns(uint64_t timeout_ns) { g_timeout_ns.store(timeout_ns > 0 ? timeout_ns : 1); }

uint64_t moe_get_launch_count(void) { return g_launches.load(); }

moe_status_t moe_set_pdl(int enable) {
    if (enable != 0 && enable != 1) return MOE_ERR_INVALID_ARG;
    g_pdl.store(enable);
    return MOE_OK;
}

moe_status_t moe_launch_events_arm(void* const* events, int n) {
    if (n < 0 || (n > 0 && !events)) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_ev.mu);
    g_ev.events.clear();
    g_ev.labels.clear();
    for (int i = 0; i < n; ++i) g_ev.events.push_back(static_cast<cudaEvent_t>(events[i]));
    g_ev_armed.store(n > 0 ? 1 : 0);
    return MOE_OK;
}

moe_status_t moe_launch_events_mark(moe_stream_t stream) {
    if (!g_ev_armed.load()) return MOE_OK;
    return cuda_status(record_next_event("mark", (cudaStream_t)stream));
}

int moe_launch_events_used(char* names, int cap) {
    std::lock_guard<std::mutex> lock(g_ev.mu);
    const int used = (int)g_ev.labels.size();
    if (names)
        for (int i = 0; i < std::min(used, cap); ++i) {
            char* dst = names + (size_t)i * MOE_LAUNCH_LABEL_BYTES;
            std::memset(dst, 0, MOE_LAUNCH_LABEL_BYTES);
            std::strncpy(dst, g_ev.labels[i].c_str(), MOE_LAUNCH_LABEL_BYTES - 1);
        }
    return used;
}

moe_status_t moe_set_gemm_pair_mode(int mode) {
    if (mode < 0 || mode > 2) return MOE_ERR_INVALID_ARG;
    g_pair_mode.store(mode);
    return MOE_OK;
}

size_t moe_workspace_size(int64_t max_T, int H, int I, int E, int S, int k, int I_shared_total) {
    if (max_T < 0 || !dim_ok(H) || !dim_ok(I) || E < 1 || E > 512 || S < 1 || S > 1024 || k < 1 || k > 32 ||
        k > E || I_shared_total < 0 || (I_shared_total > 0 && !dim_ok(I_shared_total)))
        return 0;
    const int64_t P = max_T * k;
    size_t need = route_need(max_T, H, E);
    need = std::max(need, permute_need(P, S));
    need = std::max(need, forward_layout(P, max_T, H, I, I_shared_total).total);
    // a call with fewer tokens may split the shared FC2 (fp32 partials, largest at
    // T = min(max_T, 128)) where max_T does not; every other region grows with T and P
    need = std::max(need, forward_layout(P, std::min<int64_t>(max_T, kSplitMaxT), H, I, I_shared_total).total);
    return need;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_workspace_init");
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, kWsHeaderBytes, (cudaStream_t)stream));
}

moe_status_t moe_get_device_status(void* ws, moe_stream_t stream, int32_t* device_status) {
    MOE_NVTX("moe_get_device_status");
    if (!ws || !device_status) return MOE_ERR_INVALID_ARG;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    int32_t v = 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(&v, &hdr->status, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&hdr->status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *device_status = v;
    return MOE_OK;
}

moe_status_t moe_get_route_stats(void* ws, moe_stream_t stream, int64_t* refined_tokens) {
    MOE_NVTX("moe_get_route_stats");
    if (!ws || !refined_tokens) return MOE_ERR_INVALID_ARG;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    unsigned long long v = 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(&v, &hdr->refined, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *refined_tokens = (int64_t)v;
    return MOE_OK;
}

static moe_status_t route_impl(const moe_bf16_t* x, const float* gate_w, const float* logit_bias, int64_t T, int H,
                               int E, int k, int renorm, int n_group, int topk_group, int32_t* topk_ids,
                               float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (!dim_ok(H) || E > 512 || k > 32 || T * (int64_t)k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !gate_w || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < route_need(T, H, E)) return MOE_ERR_WORKSPACE;
    const int sms = device_sms();
    RouterLaunch L;
    L.x = x;
    L.Wg = gate_w;
    L.bias = logit_bias;
    L.T = T;
    L.H = H;
    L.E = E;
    L.k = k;
    L.renorm = renorm ? 1 : 0;
    L.ids = topk_ids;
    L.w = topk_w;
    L.hdr = static_cast<WsHeader*>(ws);
    router_carve(static_cast<char*>(ws) + kWsHeaderBytes, T, E, &L.part, &L.xsq, &L.wsq);
    router_plan(T, H, E, sms, &L.nsplit, &L.KC);
    L.n_group = n_group;
    L.topk_group = topk_group;
    return cuda_status(launch_router(L, sms, (cudaStream_t)stream));
}

moe_status_t moe_route(const moe_bf16_t* x, const float* gate_w, const float* logit_bias, int64_t T, int H, int E,
                       int k, int renorm, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    MOE_NVTX("moe_route");
    return route_impl(x, gate_w, logit_bias, T, H, E, k, renorm, 1, 1, topk_ids, topk_w, ws, ws_bytes, stream);
}

moe_status_t moe_route_grouped(const moe_bf16_t* x, const float* gate_w, const float* logit_bias, int64_t T, int H,
                               int E, int k, int renorm, int n_group, int topk_group, int32_t* topk_ids,
                               float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_route_grouped");
    if (n_group < 1 || n_group > 32 || E % n_group != 0 || topk_group < 1 || topk_group > n_group ||
        k > topk_group * (E / n_group))
        return MOE_ERR_INVALID_ARG;
    return route_impl(x, gate_w, logit_bias, T, H, E, k, renorm, n_group, topk_group, topk_ids, topk_w, ws, ws_bytes,
                      stream);
}

static moe_status_t permute_impl(bool scale_rows, const int32_t* topk_ids, float* topk_w, int64_t T, int k, int E,
                                 const int32_t* rep_offset, const int32_t* rep_slots, int S, int local_start,
                                 int local_count, int nonlocal_mode, const moe_bf16_t* x, int H, int32_t* slot_ids,
                                 int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* pair_row,
                                 moe_bf16_t* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (T < 0 || k <= 0 || E <= 0 || S <= 0 || H <= 0) return MOE_ERR_INVALID_ARG;
    if (!rep_offset && S != E) return MOE_ERR_INVALID_ARG;
    if (rep_offset && !rep_slots) return MOE_ERR_INVALID_ARG;
    if (nonlocal_mode != MOE_NONLOCAL_SKIP && nonlocal_mode != MOE_NONLOCAL_MOD) return MOE_ERR_INVALID_ARG;
    if (local_count != -1 && (local_count < 1 || local_start < 0 || (int64_t)local_start + local_count > S))
        return MOE_ERR_INVALID_ARG;
    const int S_local = local_count >= 0 ? local_count : S;
    if (!dim_ok(H) || k > 32 || S_local > 1024 || T * (int64_t)k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        // an empty batch still has well-defined counts and offsets (all zero)
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)S_local, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(S_local + 1), s);
        return cuda_status(e);
    }
    if (!topk_ids || !topk_w || !slot_ids || !perm_src || !pair_row) return MOE_ERR_INVALID_ARG;
    if (x_perm && !x) return MOE_ERR_INVALID_ARG;
    if (scale_rows && !x_perm) return MOE_ERR_INVALID_ARG;
    const int64_t P = T * k;
    if (!ws || ws_bytes < permute_need(P, S_local)) return MOE_ERR_WORKSPACE;
    PermuteLaunch L;
    L.ids = topk_ids;
    L.w = topk_w;
    L.T = T;
    L.k = k;
    L.E = E;
    L.rep_offset = rep_offset;
    L.rep_slots = rep_slots;
    L.S = S;
    L.local_start = local_start;
    L.local_count = local_count;
    L.mode = nonlocal_mode;
    L.S_local = S_local;
    L.x = x;
    L.H = H;
    L.slot_ids = slot_ids;
    L.counts = counts;
    L.offsets = offsets;
    L.perm_src = perm_src;
    L.pair_row = pair_row;
    L.x_perm = x_perm;
    L.scale_rows = scale_rows;
    L.hdr = static_cast<WsHeader*>(ws);
    permute_carve(static_cast<char*>(ws) + kWsHeaderBytes, P, S_local, &L.rank, &L.chunk_cnt, &L.chunk_base);
    return cuda_status(launch_permute(L, device_sms(), s));
}

moe_status_t moe_permute(const int32_t* topk_ids, float* topk_w, int64_t T, int k, int E, const int32_t* rep_offset,
                         const int32_t* rep_slots, int S, int local_start, int local_count, int nonlocal_mode,
                         const moe_bf16_t* x, int H, int32_t* slot_ids, int32_t* counts, int32_t* offsets,
                         int32_t* perm_src, int32_t* pair_row, moe_bf16_t* x_perm, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
    MOE_NVTX("moe_permute");
    return permute_impl(false, topk_ids, topk_w, T, k, E, rep_offset, rep_slots, S, local_start, local_count,
                        nonlocal_mode, x, H, slot_ids, counts, offsets, perm_src, pair_row, x_perm, ws, ws_bytes,
                        stream);
}

moe_status_t moe_permute_on_input(const int32_t* topk_ids, float* topk_w, int64_t T, int k, int E,
                                  const int32_t* rep_offset, const int32_t* rep_slots, int S, int local_start,
                                  int local_count, int nonlocal_mode, const moe_bf16_t* x, int H, int32_t* slot_ids,
                                  int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* pair_row,
                                  moe_bf16_t* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_permute_on_input");
    return permute_impl(true, topk_ids, topk_w, T, k, E, rep_offset, rep_slots, S, local_start, local_count,
                        nonlocal_mode, x, H, slot_ids, counts, offsets, perm_src, pair_row, x_perm, ws, ws_bytes,
                        stream);
}

static moe_status_t gemm_call(bool fc1, const moe_bf16_t* a, int64_t rows_cap, const int32_t* offsets, int G,
                              const moe_bf16_t* W, int H, int I, const moe_bf16_t* a_sh, int64_t T,
                              const moe_bf16_t* Ws, int I_sh, moe_bf16_t* out, moe_bf16_t* out_sh, void* ws,
                              cudaStream_t s, float* out_sh_part = nullptr, int ksplit_sh = 1,
                              int64_t max_group_rows = -1, const float* b_scale = nullptr,
                              const float* b_scale_sh = nullptr, const float* a_scale = nullptr,
                              const float* a_scale_sh = nullptr, const int32_t* out_row = nullptr) {
    GemmLaunch L;
    L.swiglu = fc1;
    L.a = a;
    L.rows_cap = rows_cap;
    L.offsets = offsets;
    L.G = G;
    L.b = W;
    L.K = fc1 ? H : I;
    L.Nb = fc1 ? 2 * I : H;
    L.N_out = fc1 ? I : H;
    L.out = out;
    L.out_row = out_row;
    L.a_sh = a_sh;
    L.T_sh = I_sh > 0 ? T : 0;
    L.b_sh = Ws;
    L.K_sh = fc1 ? H : I_sh;
    L.Nb_sh = fc1 ? 2 * I_sh : H;
    L.N_out_sh = fc1 ? I_sh : H;
    L.out_sh = out_sh;
    L.out_sh_part = out_sh_part;
    L.ksplit_sh = ksplit_sh;
    L.hdr = static_cast<WsHeader*>(ws);
    L.timeout_ns = g_timeout_ns.load();
    L.pair_mode = g_pair_mode.load();
    // a token adds at most one row to a slot, so a group has at most T rows
    L.max_group_rows = max_group_rows >= 0 ? std::min<int64_t>(max_group_rows, rows_cap) : rows_cap;
    // E4M3 weights come with their row scales (W and Ws then point to bytes), E4M3
    // activations with theirs (a and a_sh then point to bytes)
    L.quant = a_scale ? GEMM_W8A8 : (b_scale ? GEMM_W8 : GEMM_BF16);
    L.b_scale = b_scale;
    L.b_scale_sh = b_scale_sh;
    L.a_scale = a_scale;
    L.a_scale_sh = a_scale_sh;
    const char* why = nullptr;
    return cuda_status(launch_grouped_gemm(L, device_sms(), s, &why));
}

static moe_status_t check_gemm_args(const moe_bf16_t* a, int64_t rows_cap, const int32_t* offsets, int G,
                                    const moe_bf16_t* W, int H, int I, const moe_bf16_t* a_sh, int64_t T,
                                    const moe_bf16_t* Ws, int I_sh, const moe_bf16_t* out,
                                    const moe_bf16_t* out_sh, void* ws, size_t ws_bytes) {
    if (rows_cap < 0 || G < 0 || H <= 0 || I <= 0 || T < 0 || I_sh < 0) return MOE_ERR_INVALID_ARG;
    if (!dim_ok(H) || !dim_ok(I) || (I_sh > 0 && !dim_ok(I_sh)) || G > 1024 || rows_cap >= (int64_t(1) << 31) ||
        T >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (G > 0 && rows_cap > 0 && (!a || !offsets || !W || !out)) return MOE_ERR_INVALID_ARG;
    if (I_sh > 0 && T > 0 && (!a_sh || !Ws || !out_sh)) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status_t moe_grouped_fc1(const moe_bf16_t* a, int64_t rows_cap, const int32_t* offsets, int G,
                             const moe_bf16_t* W1, int H, int I, const moe_bf16_t* a_shared, int64_t T,
                             const moe_bf16_t* W1s, int I_shared_total, moe_bf16_t* h, moe_bf16_t* h_shared,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc1");
    moe_status_t st = check_gemm_args(a, rows_cap, offsets, G, W1, H, I, a_shared, T, W1s, I_shared_total, h,
                                      h_shared, ws, ws_bytes);
    if (st != MOE_OK) return st;
    return gemm_call(true, a, rows_cap, offsets, G, W1, H, I, a_shared, T, W1s, I_shared_total, h, h_shared, ws,
                     (cudaStream_t)stream);
}

moe_status_t moe_grouped_fc2(const moe_bf16_t* h, int64_t rows_cap, const int32_t* offsets, int G,
                             const moe_bf16_t* W2, int H, int I, const moe_bf16_t* h_shared, int64_t T,
                             const moe_bf16_t* W2s, int I_shared_total, moe_bf16_t* y, moe_bf16_t* y_shared,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc2");
    moe_status_t st = check_gemm_args(h, rows_cap, offsets, G, W2, H, I, h_shared, T, W2s, I_shared_total, y,
                                      y_shared, ws, ws_bytes);
    if (st != MOE_OK) return st;
    return gemm_call(false, h, rows_cap, offsets, G, W2, H, I, h_shared, T, W2s, I_shared_total, y, y_shared, ws,
                     (cudaStream_t)stream);
}

moe_status_t moe_grouped_fc2_scatter(const moe_bf16_t* h, int64_t rows_cap, const int32_t* offsets, int G,
                                     const moe_bf16_t* W2, int H, int I, const moe_bf16_t* h_shared, int64_t T,
                                     const moe_bf16_t* W2s, int I_shared_total, const int32_t* y_row, moe_bf16_t* y,
                                     moe_bf16_t* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc2_scatter");
    moe_status_t st = check_gemm_args(h, rows_cap, offsets, G, W2, H, I, h_shared, T, W2s, I_shared_total, y,
                                      y_shared, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (rows_cap > 0 && !y_row) return MOE_ERR_INVALID_ARG;
    return gemm_call(false, h, rows_cap, offsets, G, W2, H, I, h_shared, T, W2s, I_shared_total, y, y_shared, ws,
                     (cudaStream_t)stream, nullptr, 1, -1, nullptr, nullptr, nullptr, nullptr, y_row);
}

static moe_status_t finalize_call(const moe_bf16_t* y, int64_t rows_cap, const int32_t* pair_row,
                                  const float* topk_w, int64_t T, int k, int H, const moe_bf16_t* y_shared,
                                  const float* y_shared_part, int ksplit, const moe_bf16_t* x,
                                  const moe_bf16_t* shared_gate_w, moe_bf16_t* out, void* ws, cudaStream_t s) {
    FinalizeLaunch L;
    L.y = y;
    L.rows_cap = rows_cap;
    L.pair_row = pair_row;
    L.w = topk_w;
    L.T = T;
    L.k = k;
    L.H = H;
    L.y_sh = y_shared;
    L.y_sh_part = y_shared_part;
    L.ksplit = ksplit;
    L.x = x;
    L.gate_w = shared_gate_w;
    L.out = out;
    L.hdr = static_cast<WsHeader*>(ws);
    return cuda_status(launch_finalize(L, device_sms(), s));
}

moe_status_t moe_grouped_fc1_fp8(const moe_bf16_t* a, int64_t rows_cap, const int32_t* offsets, int G,
                                 const uint8_t* W1q, const float* W1_scale, int H, int I, const moe_bf16_t* a_shared,
                                 int64_t T, const uint8_t* W1sq, const float* W1s_scale, int I_shared_total,
                                 moe_bf16_t* h, moe_bf16_t* h_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc1_fp8");
    moe_status_t st = check_gemm_args(a, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W1q), H, I,
                                      a_shared, T, reinterpret_cast<const moe_bf16_t*>(W1sq), I_shared_total, h,
                                      h_shared, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!W1_scale || (I_shared_total > 0 && T > 0 && !W1s_scale)) return MOE_ERR_INVALID_ARG;
    return gemm_call(true, a, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W1q), H, I, a_shared, T,
                     reinterpret_cast<const moe_bf16_t*>(W1sq), I_shared_total, h, h_shared, ws, (cudaStream_t)stream,
                     nullptr, 1, -1, W1_scale, W1s_scale);
}

moe_status_t moe_grouped_fc2_fp8(const moe_bf16_t* h, int64_t rows_cap, const int32_t* offsets, int G,
                                 const uint8_t* W2q, const float* W2_scale, int H, int I, const moe_bf16_t* h_shared,
                                 int64_t T, const uint8_t* W2sq, const float* W2s_scale, int I_shared_total,
                                 moe_bf16_t* y, moe_bf16_t* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc2_fp8");
    moe_status_t st = check_gemm_args(h, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W2q), H, I,
                                      h_shared, T, reinterpret_cast<const moe_bf16_t*>(W2sq), I_shared_total, y,
                                      y_shared, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!W2_scale || (I_shared_total > 0 && T > 0 && !W2s_scale)) return MOE_ERR_INVALID_ARG;
    return gemm_call(false, h, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W2q), H, I, h_shared, T,
                     reinterpret_cast<const moe_bf16_t*>(W2sq), I_shared_total, y, y_shared, ws, (cudaStream_t)stream,
                     nullptr, 1, -1, W2_scale, W2s_scale);
}

moe_status_t moe_grouped_fc1_w8a8(const uint8_t* aq, const float* a_scale, int64_t rows_cap, const int32_t* offsets,
                                  int G, const uint8_t* W1q, const float* W1_scale, int H, int I,
                                  const uint8_t* a_shared_q, const float* a_shared_scale, int64_t T, const uint8_t* W1sq,
                                  const float* W1s_scale, int I_shared_total, moe_bf16_t* h, moe_bf16_t* h_shared,
                                  void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc1_w8a8");
    const moe_bf16_t* a = reinterpret_cast<const moe_bf16_t*>(aq);
    const moe_bf16_t* a_sh = reinterpret_cast<const moe_bf16_t*>(a_shared_q);
    moe_status_t st = check_gemm_args(a, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W1q), H, I, a_sh, T,
                                      reinterpret_cast<const moe_bf16_t*>(W1sq), I_shared_total, h, h_shared, ws,
                                      ws_bytes);
    if (st != MOE_OK) return st;
    if (!W1_scale || !a_scale || (I_shared_total > 0 && T > 0 && (!W1s_scale || !a_shared_scale)))
        return MOE_ERR_INVALID_ARG;
    return gemm_call(true, a, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W1q), H, I, a_sh, T,
                     reinterpret_cast<const moe_bf16_t*>(W1sq), I_shared_total, h, h_shared, ws, (cudaStream_t)stream,
                     nullptr, 1, -1, W1_scale, W1s_scale, a_scale, a_shared_scale);
}

moe_status_t moe_grouped_fc2_w8a8(const uint8_t* hq, const float* h_scale, int64_t rows_cap, const int32_t* offsets,
                                  int G, const uint8_t* W2q, const float* W2_scale, int H, int I,
                                  const uint8_t* h_shared_q, const float* h_shared_scale, int64_t T,
                                  const uint8_t* W2sq, const float* W2s_scale, int I_shared_total, moe_bf16_t* y,
                                  moe_bf16_t* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_grouped_fc2_w8a8");
    const moe_bf16_t* a = reinterpret_cast<const moe_bf16_t*>(hq);
    const moe_bf16_t* a_sh = reinterpret_cast<const moe_bf16_t*>(h_shared_q);
    moe_status_t st = check_gemm_args(a, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W2q), H, I, a_sh, T,
                                      reinterpret_cast<const moe_bf16_t*>(W2sq), I_shared_total, y, y_shared, ws,
                                      ws_bytes);
    if (st != MOE_OK) return st;
    if (!W2_scale || !h_scale || (I_shared_total > 0 && T > 0 && (!W2s_scale || !h_shared_scale)))
        return MOE_ERR_INVALID_ARG;
    return gemm_call(false, a, rows_cap, offsets, G, reinterpret_cast<const moe_bf16_t*>(W2q), H, I, a_sh, T,
                     reinterpret_cast<const moe_bf16_t*>(W2sq), I_shared_total, y, y_shared, ws, (cudaStream_t)stream,
                     nullptr, 1, -1, W2_scale, W2s_scale, h_scale, h_shared_scale);
}

moe_status_t moe_finalize(const moe_bf16_t* y, int64_t rows_cap, const int32_t* pair_row, const float* topk_w,
                          int64_t T, int k, int H, const moe_bf16_t* y_shared, const moe_bf16_t* x,
                          const moe_bf16_t* shared_gate_w, moe_bf16_t* out, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
    MOE_NVTX("moe_finalize");
    if (T < 0 || k <= 0 || H <= 0 || rows_cap < 0) return MOE_ERR_INVALID_ARG;
    if (!dim_ok(H) || k > 32) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!pair_row || !out || (rows_cap > 0 && !y)) return MOE_ERR_INVALID_ARG;
    if (shared_gate_w && (!x || !y_shared)) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    return finalize_call(y, rows_cap, pair_row, topk_w, T, k, H, y_shared, nullptr, 0, x, shared_gate_w, out, ws,
                         (cudaStream_t)stream);
}

// moe_forward with bf16 weights (s1 == nullptr) or E4M3 weights with row scales,
// and (act8) E4M3 activations.
static moe_status_t forward_impl(const moe_bf16_t* x_perm, const int32_t* offsets, int S_local, int64_t P_cap,
                                 const void* W1, const float* s1, const void* W2, const float* s2, int H, int I,
                                 const int32_t* pair_row, const float* topk_w, int64_t T, int k,
                                 const moe_bf16_t* x, const void* W1s, const float* s1s, const void* W2s,
                                 const float* s2s, int I_shared_total, const moe_bf16_t* shared_gate_w,
                                 moe_bf16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream,
                                 bool act8 = false) {
    if (T < 0 || k <= 0 || S_local <= 0 || P_cap < 0 || H <= 0 || I <= 0 || I_shared_total < 0)
        return MOE_ERR_INVALID_ARG;
    if (!dim_ok(H) || !dim_ok(I) || (I_shared_total > 0 && !dim_ok(I_shared_total)) || k > 32 || S_local > 1024 ||
        P_cap >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    // E4M3 activations with the weights applied at the output: the token rows of x may
    // stand in for x_perm (each quantised once and placed at its pairs' rows)
    const bool from_tokens = act8 && topk_w && x;
    if ((!x_perm && !from_tokens) || !offsets || !W1 || !W2 || !pair_row || !out) return MOE_ERR_INVALID_ARG;
    if (I_shared_total > 0 && (!x || !W1s || !W2s)) return MOE_ERR_INVALID_ARG;
    if (shared_gate_w && (I_shared_total == 0 || !x)) return MOE_ERR_INVALID_ARG;
    const bool fp8 = s1 != nullptr;
    if (fp8 && (!s2 || (I_shared_total > 0 && (!s1s || !s2s)))) return MOE_ERR_INVALID_ARG;
    const ForwardLayout FL = forward_layout(P_cap, T, H, I, I_shared_total);
    if (!ws || ws_bytes < FL.total) return MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(ws);
    moe_bf16_t* h = reinterpret_cast<moe_bf16_t*>(base + FL.h);
    moe_bf16_t* h_sh = I_shared_total > 0 ? reinterpret_cast<moe_bf16_t*>(base + FL.h_sh) : nullptr;
    moe_bf16_t* y = reinterpret_cast<moe_bf16_t*>(base + FL.y);
    moe_bf16_t* y_sh = I_shared_total > 0 ? reinterpret_cast<moe_bf16_t*>(base + FL.y_sh) : nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    const int ks = shared_split(T, I, I_shared_total);
    float* y_sh_part = ks > 1 ? reinterpret_cast<float*>(base + FL.y_sh_part) : nullptr;
    moe_status_t st;
    if (act8) {
        if ((x_perm && !aligned(x_perm, 16)) || (x && !aligned(x, 16))) return MOE_ERR_INVALID_ARG;
        // E4M3 activations: quantise the expert input rows (as many as offsets[S_local]
        // says, read on the device) and the shared experts' input, run FC1 on them,
        // quantise the intermediate rows, run FC2
        const int sms = device_sms();
        const int64_t T_sh = I_shared_total > 0 ? T : 0;
        auto u8 = [&](size_t off) { return reinterpret_cast<uint8_t*>(base + off); };
        auto f32 = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
        if (from_tokens && (T > 64 || !x_perm)) {
            // weights applied at the output: the expert input rows are copies of token
            // rows, so each token row is quantised once and its codes are placed at its
            // pairs' rows (and kept for the shared experts); small batches quantise the
            // rows themselves, spread over more CTAs
            ActQuantSeg q = {x, T, nullptr, H, T_sh > 0 ? u8(FL.xsq) : nullptr, f32(FL.sxs)};
            q.pair_row = pair_row;
            q.k = k;
            q.dst2 = u8(FL.xq);
            q.scale2 = f32(FL.sxq);
            q.dst2_rows = P_cap;
            st = cuda_status(launch_quantize_act_rows(&q, 1, sms, s));
        } else {
            const ActQuantSeg qx[2] = {{x_perm, P_cap, offsets + S_local, H, u8(FL.xq), f32(FL.sxq)},
                                       {x, T_sh, nullptr, H, u8(FL.xsq), f32(FL.sxs)}};
            st = cuda_status(launch_quantize_act_rows(qx, 2, sms, s));
        }
        if (st != MOE_OK) return st;
        st = gemm_call(true, reinterpret_cast<const moe_bf16_t*>(u8(FL.xq)), P_cap, offsets, S_local,
                       static_cast<const moe_bf16_t*>(W1), H, I, reinterpret_cast<const moe_bf16_t*>(u8(FL.xsq)), T,
                       static_cast<const moe_bf16_t*>(W1s), I_shared_total, h, h_sh, ws, s, nullptr, 1, T, s1, s1s,
                       f32(FL.sxq), f32(FL.sxs));
        if (st != MOE_OK) return st;
        const ActQuantSeg qh[2] = {{h, P_cap, offsets + S_local, I, u8(FL.hq), f32(FL.shq)},
                                   {h_sh, T_sh, nullptr, I_shared_total, u8(FL.hsq), f32(FL.shs)}};
        st = cuda_status(launch_quantize_act_rows(qh, 2, sms, s));
        if (st != MOE_OK) return st;
        st = gemm_call(false, reinterpret_cast<const moe_bf16_t*>(u8(FL.hq)), P_cap, offsets, S_local,
                       static_cast<const moe_bf16_t*>(W2), H, I, reinterpret_cast<const moe_bf16_t*>(u8(FL.hsq)), T,
                       static_cast<const moe_bf16_t*>(W2s), I_shared_total, y, y_sh, ws, s, y_sh_part, ks, T, s2,
                       s2s, f32(FL.shq), f32(FL.shs));
    } else {
        st = gemm_call(true, x_perm, P_cap, offsets, S_local, static_cast<const moe_bf16_t*>(W1), H, I, x, T,
                       static_cast<const moe_bf16_t*>(W1s), I_shared_total, h, h_sh, ws, s, nullptr, 1, T, s1, s1s);
        if (st != MOE_OK) return st;
        st = gemm_call(false, h, P_cap, offsets, S_local, static_cast<const moe_bf16_t*>(W2), H, I, h_sh, T,
                       static_cast<const moe_bf16_t*>(W2s), I_shared_total, y, y_sh, ws, s, y_sh_part, ks, T, s2, s2s);
    }
    if (st != MOE_OK) return st;
    return finalize_call(y, P_cap, pair_row, topk_w, T, k, H, y_sh_part ? nullptr : y_sh, y_sh_part, ks, x,
                         shared_gate_w, out, ws, s);
}

moe_status_t moe_forward(const moe_bf16_t* x_perm, const int32_t* offsets, int S_local, int64_t P_cap,
                         const moe_bf16_t* W1, const moe_bf16_t* W2, int H, int I, const int32_t* pair_row,
                         const float* topk_w, int64_t T, int k, const moe_bf16_t* x, const moe_bf16_t* W1s,
                         const moe_bf16_t* W2s, int I_shared_total, const moe_bf16_t* shared_gate_w, moe_bf16_t* out,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_forward");
    return forward_impl(x_perm, offsets, S_local, P_cap, W1, nullptr, W2, nullptr, H, I, pair_row, topk_w, T, k, x,
                        W1s, nullptr, W2s, nullptr, I_shared_total, shared_gate_w, out, ws, ws_bytes, stream);
}

moe_status_t moe_forward_fp8(const moe_bf16_t* x_perm, const int32_t* offsets, int S_local, int64_t P_cap,
                             const uint8_t* W1q, const float* W1_scale, const uint8_t* W2q, const float* W2_scale,
                             int H, int I, const int32_t* pair_row, const float* topk_w, int64_t T, int k,
                             const moe_bf16_t* x, const uint8_t* W1sq, const float* W1s_scale, const uint8_t* W2sq,
                             const float* W2s_scale, int I_shared_total, const moe_bf16_t* shared_gate_w,
                             moe_bf16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_forward_fp8");
    if (!W1_scale || !W2_scale) return MOE_ERR_INVALID_ARG;
    return forward_impl(x_perm, offsets, S_local, P_cap, W1q, W1_scale, W2q, W2_scale, H, I, pair_row, topk_w, T, k,
                        x, W1sq, W1s_scale, W2sq, W2s_scale, I_shared_total, shared_gate_w, out, ws, ws_bytes,
                        stream);
}

moe_status_t moe_forward_w8a8(const moe_bf16_t* x_perm, const int32_t* offsets, int S_local, int64_t P_cap,
                              const uint8_t* W1q, const float* W1_scale, const uint8_t* W2q, const float* W2_scale,
                              int H, int I, const int32_t* pair_row, const float* topk_w, int64_t T, int k,
                              const moe_bf16_t* x, const uint8_t* W1sq, const float* W1s_scale, const uint8_t* W2sq,
                              const float* W2s_scale, int I_shared_total, const moe_bf16_t* shared_gate_w,
                              moe_bf16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_forward_w8a8");
    if (!W1_scale || !W2_scale) return MOE_ERR_INVALID_ARG;
    return forward_impl(x_perm, offsets, S_local, P_cap, W1q, W1_scale, W2q, W2_scale, H, I, pair_row, topk_w, T, k,
                        x, W1sq, W1s_scale, W2sq, W2s_scale, I_shared_total, shared_gate_w, out, ws, ws_bytes,
                        stream, true);
}

// longest row the NVFP4 quantiser takes (its CTA holds a row in registers)
constexpr int kNvfp4MaxK = 16384;

// One grouped GEMM on NVFP4 operands (packed E2M1 codes, E4M3 block scales, fp32
// row scales): the routed problem (A rows a, weights b per group) and the shared
// one (a_sh, b_sh).
struct Nvfp4Operands {
    const uint8_t *a, *a_sf;
    const float* a_scale;
    const uint8_t *b, *b_sf;
    const float* b_scale;
    const uint8_t *a_sh, *a_sh_sf;
    const float* a_sh_scale;
    const uint8_t *b_sh, *b_sh_sf;
    const float* b_sh_scale;
};

static moe_status_t gemm_call_nvfp4(bool fc1, const Nvfp4Operands& o, int64_t rows_cap, const int32_t* offsets,
                                    int G, int H, int I, int64_t T, int I_sh, moe_bf16_t* out, moe_bf16_t* out_sh,
                                    void* ws, cudaStream_t s, float* out_sh_part, int ksplit_sh) {
    GemmLaunch L;
    L.swiglu = fc1;
    L.a = reinterpret_cast<const uint16_t*>(o.a);
    L.rows_cap = rows_cap;
    L.offsets = offsets;
    L.G = G;
    L.b = reinterpret_cast<const uint16_t*>(o.b);
    L.K = fc1 ? H : I;
    L.Nb = fc1 ? 2 * I : H;
    L.N_out = fc1 ? I : H;
    L.out = out;
    L.a_sh = reinterpret_cast<const uint16_t*>(o.a_sh);
    L.T_sh = I_sh > 0 ? T : 0;
    L.b_sh = reinterpret_cast<const uint16_t*>(o.b_sh);
    L.K_sh = fc1 ? H : I_sh;
    L.Nb_sh = fc1 ? 2 * I_sh : H;
    L.N_out_sh = fc1 ? I_sh : H;
    L.out_sh = out_sh;
    L.out_sh_part = out_sh_part;
    L.ksplit_sh = ksplit_sh;
    L.hdr = static_cast<WsHeader*>(ws);
    L.timeout_ns = g_timeout_ns.load();
    L.pair_mode = 0;
    L.max_group_rows = std::min<int64_t>(T, rows_cap);
    L.quant = GEMM_NVFP4;
    L.b_scale = o.b_scale;
    L.b_scale_sh = o.b_sh_scale;
    L.a_scale = o.a_scale;
    L.a_scale_sh = o.a_sh_scale;
    L.a_sf = o.a_sf;
    L.a_sf_sh = o.a_sh_sf;
    L.b_sf = o.b_sf;
    L.b_sf_sh = o.b_sh_sf;
    const char* why = nullptr;
    return cuda_status(launch_grouped_gemm(L, device_sms(), s, &why));
}

moe_status_t moe_quantize_nvfp4_rows(const moe_bf16_t* v, int64_t rows, int K, int pow2, uint8_t* q, uint8_t* sb,
                                     float* scale, moe_stream_t stream) {
    MOE_NVTX("moe_quantize_nvfp4_rows");
    if (rows < 0 || K <= 0 || (pow2 != 0 && pow2 != 1)) return MOE_ERR_INVALID_ARG;
    if (K % 64 != 0 || K > kNvfp4MaxK) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!v || !q || !sb || !scale) return MOE_ERR_INVALID_ARG;
    if (!aligned(v, 16) || !aligned(q, 8)) return MOE_ERR_INVALID_ARG;
    const Nvfp4QuantSeg seg = {v, rows, nullptr, K, pow2, q, sb, scale};
    return cuda_status(launch_quantize_nvfp4_rows(&seg, 1, device_sms(), (cudaStream_t)stream));
}

moe_status_t moe_forward_nvfp4(const moe_bf16_t* x_perm, const int32_t* offsets, int S_local, int64_t P_cap,
                               const uint8_t* W1q, const uint8_t* W1_sf, const float* W1_scale, const uint8_t* W2q,
                               const uint8_t* W2_sf, const float* W2_scale, int H, int I, const int32_t* pair_row,
                               const float* topk_w, int64_t T, int k, const moe_bf16_t* x, const uint8_t* W1sq,
                               const uint8_t* W1s_sf, const float* W1s_scale, const uint8_t* W2sq,
                               const uint8_t* W2s_sf, const float* W2s_scale, int I_shared_total,
                               const moe_bf16_t* shared_gate_w, moe_bf16_t* out, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
    MOE_NVTX("moe_forward_nvfp4");
    if (T < 0 || k <= 0 || S_local <= 0 || P_cap < 0 || H <= 0 || I <= 0 || I_shared_total < 0)
        return MOE_ERR_INVALID_ARG;
    if (!dim_ok(H) || !dim_ok(I) || (I_shared_total > 0 && !dim_ok(I_shared_total)) || k > 32 || S_local > 1024 ||
        P_cap >= (int64_t(1) << 31) || H > kNvfp4MaxK || I > kNvfp4MaxK || I_shared_total > kNvfp4MaxK)
        return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!offsets || !W1q || !W1_sf || !W1_scale || !W2q || !W2_sf || !W2_scale || !pair_row || !out)
        return MOE_ERR_INVALID_ARG;
    if (I_shared_total > 0 && (!x || !W1sq || !W1s_sf || !W1s_scale || !W2sq || !W2s_sf || !W2s_scale))
        return MOE_ERR_INVALID_ARG;
    if (shared_gate_w && (I_shared_total == 0 || !x)) return MOE_ERR_INVALID_ARG;
    // weights applied at the output and the token rows given: the expert input rows are
    // copies of token rows, so each token row is quantised once and placed at its pairs'
    // rows (x_perm is then not read and may be NULL)
    const bool from_tokens = topk_w && x;
    if (!x_perm && !from_tokens) return MOE_ERR_INVALID_ARG;
    if ((!from_tokens && !aligned(x_perm, 16)) || (x && !aligned(x, 16))) return MOE_ERR_INVALID_ARG;
    const ForwardLayout FL = forward_layout(P_cap, T, H, I, I_shared_total);
    if (!ws || ws_bytes < FL.total) return MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(ws);
    auto u8 = [&](size_t off) { return reinterpret_cast<uint8_t*>(base + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
    moe_bf16_t* h = reinterpret_cast<moe_bf16_t*>(base + FL.h);
    moe_bf16_t* h_sh = I_shared_total > 0 ? reinterpret_cast<moe_bf16_t*>(base + FL.h_sh) : nullptr;
    moe_bf16_t* y = reinterpret_cast<moe_bf16_t*>(base + FL.y);
    moe_bf16_t* y_sh = I_shared_total > 0 ? reinterpret_cast<moe_bf16_t*>(base + FL.y_sh) : nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    const int ks = shared_split(T, I, I_shared_total);
    float* y_sh_part = ks > 1 ? reinterpret_cast<float*>(base + FL.y_sh_part) : nullptr;
    const int sms = device_sms();
    const int64_t T_sh = I_shared_total > 0 ? T : 0;
    // the expert input rows and the shared experts' input, to NVFP4 with power-of-two
    // row scales: per token row (placed at the shared rows and at its pairs' rows), or
    // per row of x_perm (as many as offsets[S_local] says, read on the device)
    moe_status_t st;
    if (from_tokens) {
        Nvfp4QuantSeg q = {x, T, nullptr, H, 1, T_sh > 0 ? u8(FL.xsq) : nullptr, u8(FL.xssf), f32(FL.sxs)};
        q.pair_row = pair_row;
        q.k = k;
        q.q2 = u8(FL.xq);
        q.sb2 = u8(FL.xsf);
        q.scale2 = f32(FL.sxq);
        q.dst2_rows = P_cap;
        st = cuda_status(launch_quantize_nvfp4_rows(&q, 1, sms, s));
    } else {
        const Nvfp4QuantSeg qx[2] = {{x_perm, P_cap, offsets + S_local, H, 1, u8(FL.xq), u8(FL.xsf), f32(FL.sxq)},
                                     {x, T_sh, nullptr, H, 1, u8(FL.xsq), u8(FL.xssf), f32(FL.sxs)}};
        st = cuda_status(launch_quantize_nvfp4_rows(qx, T_sh > 0 ? 2 : 1, sms, s));
    }
    if (st != MOE_OK) return st;
    const Nvfp4Operands o1 = {u8(FL.xq), u8(FL.xsf), f32(FL.sxq), W1q, W1_sf, W1_scale,
                              u8(FL.xsq), u8(FL.xssf), f32(FL.sxs), W1sq, W1s_sf, W1s_scale};
    st = gemm_call_nvfp4(true, o1, P_cap, offsets, S_local, H, I, T, I_shared_total, h, h_sh, ws, s, nullptr, 1);
    if (st != MOE_OK) return st;
    const Nvfp4QuantSeg qh[2] = {{h, P_cap, offsets + S_local, I, 1, u8(FL.hq), u8(FL.hsf), f32(FL.shq)},
                                 {h_sh, T_sh, nullptr, I_shared_total, 1, u8(FL.hsq), u8(FL.hssf), f32(FL.shs)}};
    st = cuda_status(launch_quantize_nvfp4_rows(qh, T_sh > 0 ? 2 : 1, sms, s));
    if (st != MOE_OK) return st;
    const Nvfp4Operands o2 = {u8(FL.hq), u8(FL.hsf), f32(FL.shq), W2q, W2_sf, W2_scale,
                              u8(FL.hsq), u8(FL.hssf), f32(FL.shs), W2sq, W2s_sf, W2s_scale};
    st = gemm_call_nvfp4(false, o2, P_cap, offsets, S_local, H, I, T, I_shared_total, y, y_sh, ws, s, y_sh_part, ks);
    if (st != MOE_OK) return st;
    return finalize_call(y, P_cap, pair_row, topk_w, T, k, H, y_sh_part ? nullptr : y_sh, y_sh_part, ks, x,
                         shared_gate_w, out, ws, s);
}

moe_status_t moe_quantize_act_rows(const moe_bf16_t* v, int64_t rows, int K, uint8_t* q, float* scale,
                                   moe_stream_t stream) {
    MOE_NVTX("moe_quantize_act_rows");
    if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
    if (K % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!v || !q || !scale) return MOE_ERR_INVALID_ARG;
    if (!aligned(v, 16) || !aligned(q, 8)) return MOE_ERR_INVALID_ARG;
    const ActQuantSeg seg = {v, rows, nullptr, K, q, scale};
    return cuda_status(launch_quantize_act_rows(&seg, 1, device_sms(), (cudaStream_t)stream));
}

moe_status_t moe_quantize_fp8_rows(const moe_bf16_t* w, int64_t rows, int K, uint8_t* q, float* scale,
                                   moe_stream_t stream) {
    MOE_NVTX("moe_quantize_fp8_rows");
    if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
    if (K % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!w || !q || !scale) return MOE_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(q, 8)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_fp8_rows(w, rows, K, q, scale, device_sms(), (cudaStream_t)stream));
}

moe_status_t moe_a2a_regroup(const int32_t* recv_counts, int N, int S_local, const moe_bf16_t* src, moe_bf16_t* dst,
                             int64_t rows_cap, int H, int direction, int32_t* offsets, int32_t* row_map, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_a2a_regroup");
    if (N < 1 || S_local < 1 || rows_cap < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
    if (direction != MOE_A2A_TO_GEMM && direction != MOE_A2A_TO_EXCHANGE) return MOE_ERR_INVALID_ARG;
    if ((int64_t)N * S_local > kA2aMaxBlocks || !dim_ok(H) || rows_cap > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (!recv_counts) return MOE_ERR_INVALID_ARG;
    if (rows_cap > 0 && (!src || !dst || src == dst || !aligned(src, 16) || !aligned(dst, 16)))
        return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    A2aRegroupLaunch L;
    L.recv_counts = recv_counts;
    L.N = N;
    L.S_local = S_local;
    L.rows_cap = rows_cap;
    L.H = H;
    L.src = src;
    L.dst = dst;
    L.to_exchange = direction == MOE_A2A_TO_EXCHANGE;
    L.offsets = offsets;
    L.row_map = row_map;
    L.hdr = static_cast<WsHeader*>(ws);
    return cuda_status(launch_a2a_regroup(L, device_sms(), (cudaStream_t)stream));
}

moe_status_t moe_ep_signal(int32_t* const* peer_flags, int N, int rank, int32_t epoch, moe_stream_t stream) {
    MOE_NVTX("moe_ep_signal");
    if (!peer_flags || N < 1 || N > kEpMaxRanks || rank < 0 || rank >= N) return MOE_ERR_INVALID_ARG;
    for (int n = 0; n < N; ++n)
        if (!peer_flags[n] || !aligned(peer_flags[n], 4)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_ep_signal(peer_flags, N, rank, epoch, (cudaStream_t)stream));
}

moe_status_t moe_ep_reduce(const moe_bf16_t* const* partials, int N, const int32_t* flags, int32_t epoch, int64_t row0,
                           int64_t row1, int H, moe_bf16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_NVTX("moe_ep_reduce");
    if (!partials || N < 1 || N > kEpMaxRanks || !flags || row0 < 0 || row1 < row0 || H <= 0)
        return MOE_ERR_INVALID_ARG;
    if (!dim_ok(H)) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    if (row1 == row0) return MOE_OK;
    if (!out || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    EpReduceLaunch L = {};
    for (int n = 0; n < N; ++n) {
        if (!partials[n] || !aligned(partials[n], 16)) return MOE_ERR_INVALID_ARG;
        L.partials[n] = partials[n];
    }
    L.N = N;
    L.flags = flags;
    L.epoch = epoch;
    L.row0 = row0;
    L.row1 = row1;
    L.H = H;
    L.out = out;
    L.timeout_ns = g_timeout_ns.load();
    L.hdr = static_cast<WsHeader*>(ws);
    return cuda_status(launch_ep_reduce(L, device_sms(), (cudaStream_t)stream));
}

moe_status_t moe_ipc_export(const void* ptr, uint8_t* handle, int64_t* offset) {
    MOE_NVTX("moe_ipc_export");
    if (!ptr || !handle || !offset) return MOE_ERR_INVALID_ARG;
    // cuMemGetAddressRange (driver API, version 3020): base and size of the allocation
    using RangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
    static RangeFn range_fn = nullptr;
    if (!range_fn) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 3020, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return MOE_ERR_CUDA;
        range_fn = reinterpret_cast<RangeFn>(fn);
    }
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range_fn(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS) return MOE_ERR_CUDA;
    cudaIpcMemHandle_t h;
    if (cudaIpcGetMemHandle(&h, reinterpret_cast<void*>(base)) != cudaSuccess) return MOE_ERR_CUDA;
    std::memcpy(handle, &h, sizeof(h));
    *offset = (int64_t)(reinterpret_cast<uintptr_t>(ptr) - (uintptr_t)base);
    return MOE_OK;
}

moe_status_t moe_ipc_import(const uint8_t* handle, int64_t offset, void** ptr) {
    MOE_NVTX("moe_ipc_import");
    if (!handle || !ptr || offset < 0) return MOE_ERR_INVALID_ARG;
    cudaIpcMemHandle_t h;
    std::memcpy(&h, handle, sizeof(h));
    void* base = nullptr;
    if (cudaIpcOpenMemHandle(&base, h, cudaIpcMemLazyEnablePeerAccess) != cudaSuccess) return MOE_ERR_CUDA;
    *ptr = static_cast<char*>(base) + offset;
    return MOE_OK;
}

moe_status_t moe_ipc_close(void* ptr, int64_t offset) {
    MOE_NVTX("moe_ipc_close");
    if (!ptr || offset < 0) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaIpcCloseMemHandle(static_cast<char*>(ptr) - offset));
}

moe_status_t moe_debug_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns, moe_stream_t stream) {
    if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_wait_timeout_probe(static_cast<WsHeader*>(ws), timeout_ns, (cudaStream_t)stream));
}

}  // extern "C"
