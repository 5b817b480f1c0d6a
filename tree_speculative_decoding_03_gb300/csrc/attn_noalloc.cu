// attn_noalloc.cu -- tsv_tree_verify_attn_noalloc: the tree-attention call for
// callers that cannot allocate device memory.
//
// Some callers own no allocator of their own: a plugin running inside an engine
// that hands it only its input and output buffers and keeps every other byte of
// device memory for itself, or a loop that must not call cudaMalloc because that
// call can synchronise the device.  They cannot provide the split-K workspace
// that tsv_tree_verify_attn takes.  This entry point uses instead a scratch
// array that the library itself defines in device memory, of a fixed size, so the
// call allocates nothing.
//
// The array lives for as long as the library is loaded, on every GPU that loads
// it.  All calls share it: two calls that overlap on the GPU (on different streams,
// or from different host threads) race on it, so callers must order them.  Every
// byte a call reads there (partials, per-unit records) is written earlier in the same
// call, so nothing in it needs clearing between calls.
//
// Host code cannot pass the array's name to a kernel (on the host it names a
// stand-in, not device memory): the array's device address is looked up with
// cudaGetSymbolAddress, with the device current, the first time a device's context
// calls this entry point.  The address is kept per device together with the context
// it belongs to, and looked up again if that context changes (after cudaDeviceReset
// the module, and with it the array, is loaded anew); a failed lookup is not kept.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/tsv.h"

namespace tsv {
tsv_status report_error(tsv_status s, const char* fmt, ...);
}

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

struct DeviceScratch {
    std::mutex mu;
    void* addr = nullptr;     // device address of g_attn_scratch in `ctx`
    CUcontext ctx = nullptr;  // the context the address belongs to
};
DeviceScratch g_dev[kMaxDevices];

// The calling thread's current driver context (the runtime's primary context after
// any runtime call), through the driver entry point the runtime hands out.
CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = []() -> PFN_cuCtxGetCurrent_v4000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    CUcontext c = nullptr;
    if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

}  // namespace

extern "C" size_t tsv_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" tsv_status tsv_tree_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   const int32_t* block_table, const int32_t* seq_lens,
                                                   const int32_t* parent, void* out, int B, int N, int Hq,
                                                   int Hkv, int D, int block_size, int max_blocks, int num_blocks,
                                                   float scale, tsv_dtype dtype, int32_t* seq_err, void* stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tsv::report_error(TSV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return tsv::report_error(TSV_ERR_UNSUPPORTED, "device %d beyond the %d devices supported", dev, kMaxDevices);
    const size_t need = tsv_attn_workspace_size(B, N, Hq, Hkv, D, block_size, max_blocks, dtype);
    if (need > kScratchBytes)
        return tsv::report_error(TSV_ERR_UNSUPPORTED,
                                 "tree_verify_attn_noalloc: this shape needs %zu bytes of scratch, more than the "
                                 "%zu-byte built-in array; use tsv_tree_verify_attn with a caller workspace",
                                 need, kScratchBytes);
    if (reinterpret_cast<uintptr_t>(stream) > 2) {  // not a special handle (NULL, legacy, per-thread)
        // the array used is the current device's: the stream must belong to that device
        int sdev = -1;
        e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
        if (e != cudaSuccess) return tsv::report_error(TSV_ERR_CUDA, "cudaStreamGetDevice: %s", cudaGetErrorString(e));
        if (sdev != dev)
            return tsv::report_error(TSV_ERR_ARG,
                                     "tree_verify_attn_noalloc: the stream belongs to device %d but device %d is "
                                     "current; make the stream's device current",
                                     sdev, dev);
    }
    void* scratch = nullptr;
    {
        DeviceScratch& s = g_dev[dev];
        std::lock_guard<std::mutex> lock(s.mu);
        const CUcontext ctx = current_context();
        if (s.addr == nullptr || s.ctx != ctx) {
            // set-up for this device (and context), with the device current
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_attn_scratch);
            if (e != cudaSuccess)
                return tsv::report_error(TSV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
            s.addr = p;
            s.ctx = ctx;
        }
        scratch = s.addr;
    }
    return tsv_tree_verify_attn(q, k_cache, v_cache, block_table, seq_lens, parent, out, B, N, Hq, Hkv, D,
                                block_size, max_blocks, num_blocks, scale, dtype, scratch, kScratchBytes, seq_err,
                                stream);
}
