// compact_path.cuh -- the KV-cache rewrite of one sequence's accepted path, as a block-wide
// device function shared by the compaction kernel and the verifier's fused tail.
//
// sglang report, "Tree-based Speculative Decoding (EAGLE) Implementation Summary":
// the KV cache is updated selectively for the indices of accepted tokens; SGLang
// "SpeculativeDecoding", prefix match: rejected tokens' KV is evicted.
//
// Row j of the path (1 <= j <= A) moves from logical slot L + a_j to L + j; a slot holds
// Hkv*D elements contiguously in the [num_blocks, block_size, Hkv, D] layout, so a row
// is one contiguous copy per cache (16-byte vectors).  In-place order: the source of row
// j is slot L + a_j with a_j >= j, so no row's source is the destination of an earlier
// row (nor of itself, unless a_j == j and nothing moves); the rows' vectors are therefore
// moved in increasing order a pass at a time, each pass read completely into registers
// before any of it is written.
#pragma once

#include "common.cuh"

namespace tsv {

constexpr int kCompactVecs = 8;  // 16-byte vectors one thread stages per chunk

// The cache check of block_cache_errors by one warp, without block barriers (so it can
// run while the rest of the block does other work): TSV_DERR_CAPACITY, TSV_DERR_BLOCK or 0.
__device__ __forceinline__ int warp_cache_errors(const int32_t* bt_row, int L, int N, int bs, int max_blocks,
                                                 int num_blocks) {
    if ((long long)L < 0 || (long long)L + N > (long long)max_blocks * bs) return TSV_DERR_CAPACITY;
    const int nblk = (L + N + bs - 1) / bs;
    bool bad = false;
    for (int j = (int)(threadIdx.x & 31); j < nblk; j += 32) {
        const int id = bt_row[j];
        bad |= id < 0 || id >= num_blocks;
    }
    return __any_sync(0xffffffffu, bad) ? TSV_DERR_BLOCK : 0;
}

// Checks the path 0 = a_0 < a_1 < ... < a_A < N (TSV_DERR_PARENT), then the cache
// capacity and block ids of slots [0, L + N) (TSV_DERR_CAPACITY / TSV_DERR_BLOCK), and
// moves the rows.  Returns the error (0: done).  Called by every thread of the block;
// `path` may point to global or shared memory; s_flag and s_path are shared scratch.
// block_err >= 0: the cache check was already made (its result); < 0: make it here.
__device__ __forceinline__ int compact_path(uint8_t* k_cache, uint8_t* v_cache, const int32_t* bt, int L, int A,
                                            const int32_t* path, int N, int row_bytes, int bs_log2, int max_blocks,
                                            int num_blocks, int* s_flag, int* s_path, int block_err = -1) {
    int e = 0;
    if (A > N - 1) {
        e = TSV_DERR_PARENT;
    } else {
        if (threadIdx.x == 0) *s_flag = 1;
        __syncthreads();
        for (int j = threadIdx.x; j <= A; j += blockDim.x) {
            const int a = path[j];
            s_path[j] = a;
            const bool ok = (j == 0) ? (a == 0) : (a > path[j - 1] && a < N);
            if (!ok) *s_flag = 0;
        }
        __syncthreads();
        if (!*s_flag) e = TSV_DERR_PARENT;
        __syncthreads();
    }
    if (!e) e = block_err >= 0 ? block_err : block_cache_errors(bt, L, N, 1 << bs_log2, max_blocks, num_blocks, s_flag);
    if (e) return e;
    // items (row j = 1..A, cache, vector) in increasing row order, a pass of them at a time:
    // a pass is read completely before any of it is written
    const int nvec = row_bytes >> 4;  // vectors per row and cache
    const long long total = (long long)A * 2 * nvec;
    const int pass = kCompactVecs * (int)blockDim.x;
    const long long cache_rows = (long long)num_blocks << bs_log2;
#ifdef TSV_CHECKED
    // checked build: a row index outside the cache skips the access and is reported
    if (threadIdx.x == 0) *s_flag = 0;
    __syncthreads();
    int* const bad = s_flag;
#else
    int* const bad = nullptr;
#endif
    for (long long base = 0; base < total; base += pass) {
        uint4 st[kCompactVecs];
#pragma unroll
        for (int u = 0; u < kCompactVecs; ++u) {
            const long long i = base + threadIdx.x + u * (long long)blockDim.x;
            if (i < total) {
                const int j = 1 + static_cast<int>(i / (2 * nvec)), w = static_cast<int>(i % (2 * nvec));
                const long long srow = phys_row(bt, L + s_path[j], bs_log2);
                if (!TSV_IN_BOUNDS(srow, cache_rows, bad)) continue;
                const uint8_t* cache = w < nvec ? k_cache : v_cache;
                st[u] = reinterpret_cast<const uint4*>(cache + srow * row_bytes)[w < nvec ? w : w - nvec];
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kCompactVecs; ++u) {
            const long long i = base + threadIdx.x + u * (long long)blockDim.x;
            if (i < total) {
                const int j = 1 + static_cast<int>(i / (2 * nvec)), w = static_cast<int>(i % (2 * nvec));
                const long long drow = phys_row(bt, L + j, bs_log2);
                if (s_path[j] != j && TSV_IN_BOUNDS(drow, cache_rows, bad) &&
                    TSV_IN_BOUNDS(phys_row(bt, L + s_path[j], bs_log2), cache_rows, bad)) {
                    uint8_t* cache = w < nvec ? k_cache : v_cache;
                    reinterpret_cast<uint4*>(cache + drow * row_bytes)[w < nvec ? w : w - nvec] = st[u];
                }
            }
        }
        __syncthreads();
    }
#ifdef TSV_CHECKED
    return *bad ? TSV_DERR_INTERNAL : 0;
#else
    (void)bad;
    return 0;
#endif
}

}  // namespace tsv
