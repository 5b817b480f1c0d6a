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
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/tsv.h"

namespace tsv {
tsv_status report_error(tsv_status s, const char* fmt, ...);
}

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

void* g_scratch_addr[kMaxDevices];
cudaError_t g_setup_status[kMaxDevices];
std::once_flag g_setup_once[kMaxDevices];

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
    // once per device, with that device current: the device address of the array
    std::call_once(g_setup_once[dev], [dev]() {
        g_setup_status[dev] = cudaGetSymbolAddress(&g_scratch_addr[dev], g_attn_scratch);
    });
    if (g_setup_status[dev] != cudaSuccess)
        return tsv::report_error(TSV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                                 cudaGetErrorString(g_setup_status[dev]));
    return tsv_tree_verify_attn(q, k_cache, v_cache, block_table, seq_lens, parent, out, B, N, Hq, Hkv, D,
                                block_size, max_blocks, num_blocks, scale, dtype, g_scratch_addr[dev], kScratchBytes,
                                seq_err, stream);
}
