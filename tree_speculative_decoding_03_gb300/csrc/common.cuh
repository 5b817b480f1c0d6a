// common.cuh -- small device helpers shared by the libtsv kernels.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/tsv.h"

namespace tsv {

constexpr int kMaxNodes = 128;  // tree nodes per sequence, root included

// Checked build (-DTSV_CHECKED, a test build): a global access through a computed
// index is made only if the index lies inside its buffer; otherwise TSV_DERR_INTERNAL
// is set in the given error word and the access is skipped.  The product build
// compiles the checks away (the condition is not evaluated).
__device__ __forceinline__ bool checked_in_bounds(long long i, long long n, int32_t* err) {
    if (i >= 0 && i < n) return true;
    if (err != nullptr) atomicOr(err, TSV_DERR_INTERNAL);
    return false;
}
#ifdef TSV_CHECKED
#define TSV_IN_BOUNDS(idx, extent, errp) (::tsv::checked_in_bounds((long long)(idx), (long long)(extent), (errp)))
#else
#define TSV_IN_BOUNDS(idx, extent, errp) true
#endif

// Programmatic dependent launch: every kernel of the library lets the next kernel in the
// stream start launching early (pdl_launch_dependents) and waits for the previous one to
// complete, with its writes visible, before reading anything (pdl_wait).  Without the
// launch attribute both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kernel` with programmatic stream serialisation (it may start while the
// previous kernel in the stream finishes; it waits for it with pdl_wait), plus an
// optional cluster shape.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster_x > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Validates one sequence's tree: parent[0] == -1 and 0 <= parent[i] < i.
// Cooperative over the calling block; every thread gets the same answer.
__device__ __forceinline__ bool block_tree_ok(const int32_t* par, int N, int* s_flag) {
    if (threadIdx.x == 0) *s_flag = 1;
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        int p = par[i];
        bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
        if (!ok) *s_flag = 0;
    }
    __syncthreads();
    bool r = *s_flag != 0;
    __syncthreads();
    return r;
}

// Capacity and block-id checks for logical slots [0, L + N) of one sequence;
// returns TSV_DERR_CAPACITY, TSV_DERR_BLOCK or 0 (capacity is checked first).
__device__ __forceinline__ int block_cache_errors(const int32_t* bt_row, int L, int N, int bs,
                                                  int max_blocks, int num_blocks, int* s_flag) {
    if ((long long)L < 0 || (long long)L + N > (long long)max_blocks * bs) return TSV_DERR_CAPACITY;
    if (threadIdx.x == 0) *s_flag = 0;
    __syncthreads();
    int nblk = (L + N + bs - 1) / bs;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
        int id = bt_row[j];
        if (id < 0 || id >= num_blocks) *s_flag = TSV_DERR_BLOCK;
    }
    __syncthreads();
    int r = *s_flag;
    __syncthreads();
    return r;
}

// Ancestor masks of the tree: anc[n] (4 x 32 bits) has bit j set iff node j is on the
// root-to-n path, n included.  Threads n < N each walk up their own path; the walk is
// bounded by N steps, so an invalid parent array cannot make it loop.
__device__ __forceinline__ void build_ancestor_masks(const int32_t* par, int N, uint32_t (*anc)[4]) {
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        uint32_t m[4] = {0u, 0u, 0u, 0u};
        int a = n;
        for (int step = 0; step <= N && a >= 0 && a < N; ++step) {
            m[a >> 5] |= 1u << (a & 31);
            a = par[a];
        }
        anc[n][0] = m[0];
        anc[n][1] = m[1];
        anc[n][2] = m[2];
        anc[n][3] = m[3];
    }
}

__device__ __forceinline__ bool anc_has(const uint32_t* m, int j) { return (m[j >> 5] >> (j & 31)) & 1u; }

// Writes the tree's new K/V rows of sequence b (k_new / v_new [B, N, Hkv, D], one
// row = row_bytes contiguous bytes: all kv heads of a node) into the paged caches at
// logical slots L .. L + N - 1, in 16-byte vectors (row_bytes is a multiple of 16 and
// every base is 16-byte aligned).  The block ids covering [0, L + N) must have been
// checked.  Cooperative over the calling block.  cache_vecs / new_vecs: 16-byte vectors
// in a cache / in k_new (the checked build's bounds); err: the sequence's error word.
__device__ __forceinline__ void append_tree_rows(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                                 const int32_t* bt_row, int b, int L, int N, int row_bytes,
                                                 int bs_log2, long long cache_vecs, long long new_vecs,
                                                 int32_t* err) {
    const int vecs = row_bytes >> 4;  // 16-byte vectors per row
    const long long src0 = (long long)b * N * vecs;
    const int total = 2 * N * vecs;     // K rows first, then V rows
    constexpr int U = 4;                // vectors in flight per thread
    for (int base = 0; base < total; base += U * (int)blockDim.x) {
        uint4 val[U];
        long long dst[U];
        int kvs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = base + u * (int)blockDim.x + (int)threadIdx.x;
            kvs[u] = -1;
            if (idx < total) {
                const int kv = idx >= N * vecs;
                const int r = kv ? idx - N * vecs : idx;
                const int j = r / vecs, c = r - j * vecs;
                const int t = L + j;
                dst[u] = ((long long)bt_row[t >> bs_log2] * (1 << bs_log2) + (t & ((1 << bs_log2) - 1))) * vecs + c;
                if (!TSV_IN_BOUNDS(dst[u], cache_vecs, err) || !TSV_IN_BOUNDS(src0 + (long long)j * vecs + c, new_vecs, err))
                    continue;
                val[u] = __ldg(static_cast<const uint4*>(kv ? v_new : k_new) + src0 + (long long)j * vecs + c);
                kvs[u] = kv;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (kvs[u] >= 0) static_cast<uint4*>(kvs[u] ? v_cache : k_cache)[dst[u]] = val[u];
    }
}

// Physical row of logical slot t (block ids already validated by the caller).
__device__ __forceinline__ long long phys_row(const int32_t* bt_row, int t, int bs_log2) {
    return (long long)bt_row[t >> bs_log2] * (1 << bs_log2) + (t & ((1 << bs_log2) - 1));
}

}  // namespace tsv
