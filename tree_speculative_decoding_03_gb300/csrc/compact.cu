// compact.cu -- KV-cache rewrite of the accepted root-to-leaf path.
//
// sglang report, "Tree-based Speculative Decoding (EAGLE) Implementation Summary":
// the KV cache is updated selectively for the indices of accepted tokens, and
// "Issue: Speculative Decoding on vLLM": trees require this rewrite.  SGLang
// "SpeculativeDecoding", prefix match: rejected tokens' KV is evicted.
//
// One CTA per sequence.  A slot holds Hkv*D elements contiguously in the
// [num_blocks, block_size, Hkv, D] layout, so moving one path row is one
// contiguous copy per cache, done with 16-byte vector loads/stores.  Path rows
// are moved in increasing j with a barrier after each: the source of row j is
// slot L + a_j with a_j >= j, so it can be the destination of a later row
// (a_j == j' > j) but never of an earlier one -- copying in order, each row fully
// read before the next is written, is the in-place safe order.
#include "common.cuh"

namespace tsv {

__global__ void __launch_bounds__(256) kv_compact_kernel(
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ accepted_nodes,
    const int32_t* __restrict__ accept_len, int32_t* __restrict__ new_seq_lens, int N, int row_bytes,
    int bs_log2, int max_blocks, int num_blocks, int32_t* __restrict__ seq_err) {
    __shared__ int s_flag;
    __shared__ int s_path[kMaxNodes];
    pdl_wait();  // accepted paths come from the previous kernel
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int L = seq_lens[b];
    const int A = accept_len[b];
    if (A < 0) {
        if (threadIdx.x == 0) {
            new_seq_lens[b] = L;
            seq_err[b] = 0;
        }
        return;
    }
    const int32_t* path = accepted_nodes + (long long)b * N;
    int e = 0;
    if (A > N - 1) {
        e = TSV_DERR_PARENT;
    } else {
        if (threadIdx.x == 0) s_flag = 1;
        __syncthreads();
        for (int j = threadIdx.x; j <= A; j += blockDim.x) {
            int a = path[j];
            s_path[j] = a;
            bool ok = (j == 0) ? (a == 0) : (a > path[j - 1] && a < N);
            if (!ok) s_flag = 0;
        }
        __syncthreads();
        if (!s_flag) e = TSV_DERR_PARENT;
        __syncthreads();
    }
    const int32_t* bt = block_table + (long long)b * max_blocks;
    if (!e) e = block_cache_errors(bt, L, N, 1 << bs_log2, max_blocks, num_blocks, &s_flag);
    if (e) {
        if (threadIdx.x == 0) {
            seq_err[b] = e;
            new_seq_lens[b] = L;
        }
        return;
    }
    const int nvec = row_bytes >> 4;
    for (int j = 1; j <= A; ++j) {
        const int a = s_path[j];
        if (a != j) {
            const long long src = phys_row(bt, L + a, bs_log2) * row_bytes;
            const long long dst = phys_row(bt, L + j, bs_log2) * row_bytes;
            const uint4* ks = reinterpret_cast<const uint4*>(k_cache + src);
            const uint4* vs = reinterpret_cast<const uint4*>(v_cache + src);
            uint4* kd = reinterpret_cast<uint4*>(k_cache + dst);
            uint4* vd = reinterpret_cast<uint4*>(v_cache + dst);
            for (int i = threadIdx.x; i < 2 * nvec; i += blockDim.x) {
                if (i < nvec) {
                    kd[i] = ks[i];
                } else {
                    vd[i - nvec] = vs[i - nvec];
                }
            }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        new_seq_lens[b] = L + 1 + A;
        seq_err[b] = 0;
    }
}

cudaError_t launch_kv_compact(void* k_cache, void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* accepted_nodes, const int32_t* accept_len, int32_t* new_seq_lens,
                              int B, int N, int Hkv, int D, int block_size, int max_blocks, int num_blocks,
                              int elem_bytes, int32_t* seq_err, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    int bs_log2 = 0;
    while ((1 << bs_log2) < block_size) ++bs_log2;
    return launch_pdl(kv_compact_kernel, dim3(static_cast<unsigned>(B)), dim3(256), 0, stream, 1u,
                      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), block_table, seq_lens,
                      accepted_nodes, accept_len, new_seq_lens, N, Hkv * D * elem_bytes, bs_log2, max_blocks,
                      num_blocks, seq_err);
}

}  // namespace tsv
