// attn_tc.cu -- placeholder until the tensor-core path lands.
#include "attn_common.cuh"
namespace tsv {
bool attn_tc_supported(int) { return false; }
int attn_tc_rows_per_cta() { return 256; }
cudaError_t launch_attn_tc(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace tsv
