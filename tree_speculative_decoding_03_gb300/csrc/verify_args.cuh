// verify_args.cuh -- arguments of the rejection-sampling kernel (see verify.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tsv {

struct SampleArgs {
    const float* logits;
    const float* probs;
    const int32_t* tokens;
    const int32_t* parent;
    const float* u_accept;
    const float* u_bonus;
    float T;
    int N;
    int V;
    int v_per_cta;  // vocabulary entries owned by one CTA (multiple of 4); set by the launcher
    int32_t* accepted_nodes;
    int32_t* accept_len;
    int32_t* bonus_token;
    int32_t* out_tokens;
    int32_t* seq_err;
};

cudaError_t launch_tree_reject(SampleArgs a, int B, int num_sms, cudaStream_t stream);

}  // namespace tsv
