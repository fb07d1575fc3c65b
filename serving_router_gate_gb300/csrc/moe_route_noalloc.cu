// moe_route_noalloc.cu -- moe_route for callers that cannot allocate device
// memory.
//
// moe_route needs a caller-provided workspace for its partial logits.  Some
// callers cannot provide one: a plugin that a host framework hands only its
// input and output buffers, a runtime whose device memory is owned by a pool
// this library cannot reach, or a deployment that forbids device allocation
// once it is serving.  moe_route_noalloc runs the same two router kernels with
// their scratch in a fixed-size array that lives in this library's own device
// memory, so the caller passes inputs and outputs only.
//
// The array: kNoallocScratchBytes (16 MiB) of file-scope __device__ memory.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks its address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should therefore come before any
// stream capture.  Every call uses the same array and overwrites every entry
// it later reads, so nothing has to be cleared between calls.  Calls that
// overlap on one device (on two streams, or two graph replays in flight) race
// on it; calls ordered on one stream do not, and calls on different devices
// use separate copies of the array.
#include <algorithm>
#include <mutex>

#include "moe_internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

// Device address of g_route_scratch and the SM count of the current device,
// looked up once per device.
moe_status_t device_scratch(void** ptr, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return MOE_ERR_CUDA;
        g_scratch[dev] = p;
        g_sms[dev] = n;
    }
    *ptr = g_scratch[dev];
    *sms = g_sms[dev];
    return MOE_OK;
}

// Bytes of scratch for a K split into `nsplit` ranges.
size_t scratch_bytes(int64_t T, int E, int nsplit) {
    return up256((size_t)nsplit * (size_t)T * (size_t)E * sizeof(float)) +
           up256((size_t)nsplit * (size_t)T * sizeof(float)) + up256((size_t)nsplit * (size_t)E * sizeof(float));
}

}  // namespace

extern "C" MOE_API moe_status_t moe_route_noalloc(const moe_bf16_t* x, const float* gate_w, const float* logit_bias,
                                                  int64_t T, int H, int E, int k, int renorm, int32_t* topk_ids,
                                                  float* topk_w, moe_stream_t stream) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (H % 64 != 0 || H > (1 << 20) || E > 512 || k > 32 || T * (int64_t)k >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !gate_w || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    // the smallest possible scratch (one K range) must fit in the array
    if (scratch_bytes(T, E, 1) > kNoallocScratchBytes) return MOE_ERR_UNSUPPORTED;

    void* base = nullptr;
    int sms = 0;
    moe_status_t st = device_scratch(&base, &sms);
    if (st != MOE_OK) return st;

    // the split moe_route would use, reduced until its scratch fits the array.  Each
    // pass lowers nsplit by at least one (ranges of ceil(H / (nsplit - 1)) rounded up
    // to 32), so the loop ends with a layout that fits: either the test failed, or
    // nsplit reached 1, whose size was checked above.
    int nsplit = 1, KC = H;
    moe::router_plan(T, H, E, sms, &nsplit, &KC);
    while (nsplit > 1 && scratch_bytes(T, E, nsplit) > kNoallocScratchBytes) {
        int kc = (H + nsplit - 2) / (nsplit - 1);
        kc = (kc + 31) / 32 * 32;
        KC = kc;
        nsplit = (H + kc - 1) / kc;
    }

    moe::RouterLaunch L;
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
    L.nsplit = nsplit;
    L.KC = KC;
    L.hdr = nullptr;  // no workspace header: the refined-token counter is not kept
    char* p = static_cast<char*>(base);
    L.part = reinterpret_cast<float*>(p);
    L.xsq = reinterpret_cast<float*>(p + up256((size_t)nsplit * (size_t)T * (size_t)E * sizeof(float)));
    L.wsq = reinterpret_cast<float*>(reinterpret_cast<char*>(L.xsq) + up256((size_t)nsplit * (size_t)T * sizeof(float)));
    return moe::launch_router(L, sms, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
