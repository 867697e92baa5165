// mla_sparse_decode_static_ws: the same decode as mla_sparse_decode, for
// callers that cannot allocate device memory themselves.
//
// Some callers have no allocator to draw from: plugin hosts that own every
// device buffer and give extensions only the tensors they pass in,
// latency-critical serving loops that forbid allocator calls (a cudaMalloc
// may synchronise the device), and code whose memory plan is fixed ahead of
// time.  They can still hand over inputs and outputs, but not a workspace.
// This entry point takes its scratch from one fixed array that lives in this
// library's device image instead.
#include "common.cuh"
#include "kernels.cuh"

#include <cuda.h>

#include <mutex>

namespace {

// Scratch shared by every call of mla_sparse_decode_static_ws on a device.
// It is part of the library's device image: each GPU that loads the library
// keeps these MLA_STATIC_WS_BYTES reserved until the process exits.
static __device__ __align__(256) unsigned char g_static_ws[MLA_STATIC_WS_BYTES];

// Device address of g_static_ws per device.  The name g_static_ws in host
// code is only a host-side stand-in, so the address is looked up with that
// device current.  The lookup is cached together with the context it was
// made in: after cudaDeviceReset (or any re-creation of the primary context)
// the library's device image is loaded again, possibly at another address,
// and the next call looks the address up afresh.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q{};
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

struct StaticWsAddr {
    std::mutex mu;
    void *ptr[64] = {};
    CUcontext ctx[64] = {};
};

StaticWsAddr &addr_table() {
    static StaticWsAddr t;
    return t;
}

int static_ws_ptr(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MLA_ERR_DEVICE;
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) return MLA_ERR_CUDA;
    StaticWsAddr &t = addr_table();
    std::lock_guard<std::mutex> lock(t.mu);
    if (!ctx || !t.ptr[dev] || t.ctx[dev] != ctx) {
        // the lookup also makes the device's primary context current when no
        // context is yet; the context is named after it
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return MLA_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return MLA_ERR_CUDA;
        t.ptr[dev] = p;
        t.ctx[dev] = ctx;
    }
    *out = t.ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" int mla_sparse_decode_static_ws(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                                           int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int B,
                                           float softmax_scale, const mla_bf16 *wkv_b, float *out,
                                           int32_t *dev_status, mla_stream_t stream) {
    const size_t need = mla_sparse_decode_workspace_size(B, K);
    if (need == 0 || need > MLA_STATIC_WS_BYTES) return MLA_ERR_SIZE;
    void *ws = nullptr;
    const int rc = static_ws_ptr(&ws);
    if (rc != MLA_OK) return rc;
    // nothing in the scratch has to start at zero: every byte the kernels read
    // is written earlier in the same call
    return mla_sparse_decode(q_lat, kv_cache, pe_cache, S_cap, topk_idx, K, end_pos, B, softmax_scale, wkv_b, out, ws,
                             MLA_STATIC_WS_BYTES, dev_status, stream);
}
