// verify_args.cuh -- arguments of the rejection-sampling kernel (see verify.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tsv {

struct SampleArgs {
    const void* logits;  // [B, N, V] fp32, or bf16 when logits_bf16
    const float* probs;
    const int32_t* tokens;
    const int32_t* parent;
    const float* u_accept;
    const float* u_bonus;
    float T;
    int replacement;  // siblings drafted independently from q (with replacement): q is never updated
    int top_k;        // > 0: target filtered to its top_k tokens at every visited node
    float top_p;      // < 1: target filtered to the smallest top set of mass >= top_p
    int logits_bf16;
    int N;
    int V;
    int v_per_cta;  // vocabulary entries owned by one CTA (multiple of 4); set by the launcher
    int32_t* accepted_nodes;
    int32_t* accept_len;
    int32_t* bonus_token;
    int32_t* out_tokens;
    int32_t* seq_err;
    // fused KV-cache rewrite of the accepted path (k_cache == nullptr: none); same
    // arguments and results as the compaction kernel, errors in compact_err
    uint8_t* k_cache;
    uint8_t* v_cache;
    const int32_t* block_table;
    const int32_t* seq_lens;
    int32_t* new_seq_lens;
    int32_t* compact_err;
    int row_bytes, bs_log2, max_blocks, num_blocks;
};

cudaError_t launch_tree_reject(SampleArgs a, int B, int num_sms, cudaStream_t stream);

}  // namespace tsv
