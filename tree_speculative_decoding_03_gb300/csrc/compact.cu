// compact.cu -- KV-cache rewrite of the accepted root-to-leaf path.
//
// sglang report, "Tree-based Speculative Decoding (EAGLE) Implementation Summary":
// the KV cache is updated selectively for the indices of accepted tokens, and
// "Issue: Speculative Decoding on vLLM": trees require this rewrite.  SGLang
// "SpeculativeDecoding", prefix match: rejected tokens' KV is evicted.
//
// One CTA per sequence; the rewrite itself is compact_path (compact_path.cuh), which
// the verifier's fused tail runs too.
#include "compact_path.cuh"

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
    const int e = compact_path(k_cache, v_cache, block_table + (long long)b * max_blocks, L, A,
                               accepted_nodes + (long long)b * N, N, row_bytes, bs_log2, max_blocks, num_blocks,
                               &s_flag, s_path);
    if (threadIdx.x == 0) {
        seq_err[b] = e;
        new_seq_lens[b] = e ? L : L + 1 + A;
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
