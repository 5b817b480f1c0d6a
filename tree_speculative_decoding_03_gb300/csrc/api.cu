// api.cu -- the C ABI of libtsv: host-side argument checks, launch planning and
// dispatch to the kernels.  No allocation, no host synchronisation.
#include <cstdarg>
#include <cstdio>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {
cudaError_t launch_kv_compact(void* k_cache, void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* accepted_nodes, const int32_t* accept_len, int32_t* new_seq_lens,
                              int B, int N, int Hkv, int D, int block_size, int max_blocks, int num_blocks,
                              int elem_bytes, int32_t* seq_err, cudaStream_t stream);
cudaError_t launch_attn_simt_f32(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_merge(const AttnArgs& a, bool bf16, cudaStream_t stream);
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream);
bool attn_tc_supported(int D);
int attn_tc_rows_per_cta();
}  // namespace tsv

#include "verify_args.cuh"

namespace {

thread_local char g_err[512] = "";

tsv_status fail(tsv_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

tsv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TSV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
    return sms;
}

bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int log2i(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

bool use_tc(tsv_dtype dt, int D) { return dt == TSV_BF16 && tsv::attn_tc_supported(D); }  // D checked before

tsv::AttnPlan plan_for(int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks, tsv_dtype dt) {
    // tensor-core path: persistent CTAs, one per SM, splitting all tiles evenly; FMA
    // work items are small: eight waves of key chunks of at least 256 keys
    if (use_tc(dt, D))
        return tsv::make_attn_plan_tc(B, N, Hq, Hkv, D, block_size, max_blocks, tsv::attn_tc_rows_per_cta(),
                                      device_sms());
    return tsv::make_attn_plan(B, N, Hq, Hkv, D, block_size, max_blocks, 16, device_sms(), 8, 256);
}

tsv_status check_attn_shapes(int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                             int num_blocks, tsv_dtype dt) {
    if (B < 0 || N < 1 || Hq < 1 || Hkv < 1 || max_blocks < 1 || num_blocks < 1)
        return fail(TSV_ERR_ARG, "bad sizes B=%d N=%d Hq=%d Hkv=%d max_blocks=%d num_blocks=%d", B, N, Hq, Hkv,
                    max_blocks, num_blocks);
    if (Hq % Hkv) return fail(TSV_ERR_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (N > tsv::kMaxNodes) return fail(TSV_ERR_UNSUPPORTED, "N=%d exceeds %d tree nodes", N, tsv::kMaxNodes);
    if (D != 64 && D != 128) return fail(TSV_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", D);
    if (!pow2_in(block_size, 8, 128)) return fail(TSV_ERR_UNSUPPORTED, "block_size %d not a power of two in [8,128]", block_size);
    if (dt != TSV_BF16 && dt != TSV_F32) return fail(TSV_ERR_ARG, "bad dtype %d", (int)dt);
    if ((long long)N * (Hq / Hkv) > 1024) return fail(TSV_ERR_UNSUPPORTED, "N * Hq / Hkv = %d > 1024 rows", N * (Hq / Hkv));
    return TSV_OK;
}

}  // namespace

namespace tsv {
// Records a failure message for tsv_last_error() from other translation units.
tsv_status report_error(tsv_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace tsv

extern "C" {

const char* tsv_last_error(void) { return g_err; }

size_t tsv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                               tsv_dtype dtype) {
    if (check_attn_shapes(B, N, Hq, Hkv, D, block_size, max_blocks, 1, dtype) != TSV_OK) return 0;
    return plan_for(B, N, Hq, Hkv, D, block_size, max_blocks, dtype).ws_bytes;
}

}  // extern "C"

namespace {
// The attention call, with the fused append of the tree's rows when k_new != nullptr.
tsv_status verify_attn(const void* q, const void* k_new, const void* v_new, void* k_cache_w, void* v_cache_w,
                       const void* k_cache, const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                       const int32_t* parent, void* out, int B, int N, int Hq, int Hkv, int D, int block_size,
                       int max_blocks, int num_blocks, float scale, tsv_dtype dtype, void* workspace,
                       size_t workspace_bytes, int32_t* seq_err, void* stream) {
    tsv_status st = check_attn_shapes(B, N, Hq, Hkv, D, block_size, max_blocks, num_blocks, dtype);
    if (st != TSV_OK) return st;
    if (B == 0) return TSV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !parent || !out || !seq_err)
        return fail(TSV_ERR_ARG, "null array argument");
    if (k_new != nullptr && (!v_new || !aligned16(k_new) || !aligned16(v_new)))
        return fail(TSV_ERR_ARG, "k_new and v_new must be non-null and 16-byte aligned");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(TSV_ERR_ARG, "q, caches and out must be 16-byte aligned");
    if (!(scale > 0.0f) || !isfinite(scale)) return fail(TSV_ERR_ARG, "scale must be positive and finite");
    const tsv::AttnPlan p = plan_for(B, N, Hq, Hkv, D, block_size, max_blocks, dtype);
    if (p.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < p.ws_bytes))
        return fail(TSV_ERR_ARG, "workspace of %zu bytes needed, %zu given", p.ws_bytes, workspace_bytes);
    if (p.ws_bytes > 0 && !aligned16(workspace)) return fail(TSV_ERR_ARG, "workspace must be 16-byte aligned");

    tsv::AttnArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache_w = k_cache_w;
    a.v_cache_w = v_cache_w;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.parent = parent;
    a.out = out;
    const bool tc = use_tc(dtype, D);
    // partial rows: tensor-core path two slots per CTA, FMA path one per (b, g, chunk)
    const size_t rows = tc ? 2 * (size_t)p.lanes * p.n_rgroups * p.rows_item : (size_t)B * Hkv * p.max_chunks * p.R;
    a.part_o = static_cast<float*>(workspace);
    a.part_m = p.ws_bytes ? a.part_o + rows * D : nullptr;
    a.part_l = p.ws_bytes ? a.part_m + rows : nullptr;
    a.unit_info = (tc && p.ws_bytes) ? reinterpret_cast<int*>(a.part_l + rows) : nullptr;
    a.lanes = p.lanes;
    a.rows_item = p.rows_item;
    a.seq_err = seq_err;
    a.B = B;
    a.N = N;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.bs_log2 = log2i(block_size);
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.G = p.G;
    a.R = p.R;
    a.rows_per_cta = p.rows_per_cta;
    a.n_rgroups = p.n_rgroups;
    a.chunk = p.chunk;
    a.max_chunks = p.max_chunks;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tc) {
        e = tsv::launch_attn_tc(a, s);  // check kernel, persistent kernel, merge kernel
    } else {
        e = tsv::launch_attn_simt_f32(a, s);
        if (e == cudaSuccess) e = tsv::launch_attn_merge(a, false, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "tree_verify_attn launch");
    return TSV_OK;
}
}  // namespace

extern "C" {

tsv_status tsv_tree_verify_attn(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, const int32_t* parent,
                                void* out, int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                                int num_blocks, float scale, tsv_dtype dtype, void* workspace,
                                size_t workspace_bytes, int32_t* seq_err, void* stream) {
    return verify_attn(q, nullptr, nullptr, nullptr, nullptr, k_cache, v_cache, block_table, seq_lens, parent, out, B,
                       N, Hq, Hkv, D, block_size, max_blocks, num_blocks, scale, dtype, workspace, workspace_bytes,
                       seq_err, stream);
}

tsv_status tsv_tree_verify_attn_append(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                                       const int32_t* parent, void* out, int B, int N, int Hq, int Hkv, int D,
                                       int block_size, int max_blocks, int num_blocks, float scale, tsv_dtype dtype,
                                       void* workspace, size_t workspace_bytes, int32_t* seq_err, void* stream) {
    if (B > 0 && (!k_new || !v_new)) return fail(TSV_ERR_ARG, "null k_new / v_new");
    return verify_attn(q, k_new, v_new, k_cache, v_cache, k_cache, v_cache, block_table, seq_lens, parent, out, B, N,
                       Hq, Hkv, D, block_size, max_blocks, num_blocks, scale, dtype, workspace, workspace_bytes, seq_err,
                       stream);
}

}  // extern "C"

namespace {
// Argument checks and packing shared by the walk alone and the walk with fused compaction.
tsv_status reject_args(const void* target_logits, const float* draft_probs, const int32_t* draft_tokens,
                       const int32_t* parent, const float* u_accept, const float* u_bonus, float temperature, int B,
                       int N, int V, int32_t* accepted_nodes, int32_t* accept_len, int32_t* bonus_token,
                       int32_t* out_tokens, int32_t* seq_err, const tsv_walk_options* opts, tsv::SampleArgs* a) {
    const tsv_walk_options o = opts ? *opts : tsv_walk_options{0, TSV_F32, 0, 1.0f};
    if (o.with_replacement != 0 && o.with_replacement != 1)
        return fail(TSV_ERR_ARG, "with_replacement must be 0 or 1, not %d", o.with_replacement);
    if (o.logits_dtype != TSV_F32 && o.logits_dtype != TSV_BF16)
        return fail(TSV_ERR_ARG, "bad logits dtype %d", (int)o.logits_dtype);
    if (o.top_k < 0 || !(o.top_p > 0.0f && o.top_p <= 1.0f))
        return fail(TSV_ERR_ARG, "top_k must be >= 0 and top_p in (0, 1]");
    if (B < 0 || N < 1 || V < 1) return fail(TSV_ERR_ARG, "bad sizes B=%d N=%d V=%d", B, N, V);
    if (N > tsv::kMaxNodes) return fail(TSV_ERR_UNSUPPORTED, "N=%d exceeds %d tree nodes", N, tsv::kMaxNodes);
    if (V > 16 * 512 * 32) return fail(TSV_ERR_UNSUPPORTED, "V=%d exceeds %d", V, 16 * 512 * 32);
    if (!(temperature >= 0.0f) || !isfinite(temperature)) return fail(TSV_ERR_ARG, "temperature must be finite and >= 0");
    if (temperature > 0.0f && temperature < 1e-6f)
        return fail(TSV_ERR_UNSUPPORTED, "temperature %g in (0, 1e-6): use 0 for greedy matching", temperature);
    const bool greedy = temperature == 0.0f;
    if (B > 0 && (!target_logits || !draft_tokens || !parent || !accepted_nodes || !accept_len || !bonus_token ||
                  !out_tokens || !seq_err || (!greedy && (!draft_probs || !u_accept || !u_bonus))))
        return fail(TSV_ERR_ARG, "null array argument");
    *a = tsv::SampleArgs{};
    a->logits = target_logits;
    a->probs = greedy ? nullptr : draft_probs;
    a->tokens = draft_tokens;
    a->parent = parent;
    a->u_accept = u_accept;
    a->u_bonus = u_bonus;
    a->T = temperature;
    a->replacement = o.with_replacement;
    a->top_k = o.top_k;
    a->top_p = o.top_p;
    a->logits_bf16 = o.logits_dtype == TSV_BF16;
    a->N = N;
    a->V = V;
    a->accepted_nodes = accepted_nodes;
    a->accept_len = accept_len;
    a->bonus_token = bonus_token;
    a->out_tokens = out_tokens;
    a->seq_err = seq_err;
    return TSV_OK;
}

tsv_status compact_args(void* k_cache, void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                        int32_t* new_seq_lens, int B, int N, int Hkv, int D, int block_size, int max_blocks,
                        int num_blocks, tsv_dtype dtype, int32_t* seq_err) {
    if (B < 0 || N < 1 || Hkv < 1 || max_blocks < 1 || num_blocks < 1)
        return fail(TSV_ERR_ARG, "bad sizes B=%d N=%d Hkv=%d", B, N, Hkv);
    if (N > tsv::kMaxNodes) return fail(TSV_ERR_UNSUPPORTED, "N=%d exceeds %d tree nodes", N, tsv::kMaxNodes);
    if (D != 64 && D != 128) return fail(TSV_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", D);
    if (!pow2_in(block_size, 8, 128)) return fail(TSV_ERR_UNSUPPORTED, "block_size %d not a power of two in [8,128]", block_size);
    if (dtype != TSV_BF16 && dtype != TSV_F32) return fail(TSV_ERR_ARG, "bad dtype %d", (int)dtype);
    if (B > 0 && (!k_cache || !v_cache || !block_table || !seq_lens || !new_seq_lens || !seq_err))
        return fail(TSV_ERR_ARG, "null array argument");
    if (B > 0 && (!aligned16(k_cache) || !aligned16(v_cache))) return fail(TSV_ERR_ARG, "caches must be 16-byte aligned");
    return TSV_OK;
}
}  // namespace

extern "C" {

tsv_status tsv_tree_reject_sample_ex(const void* target_logits, const float* draft_probs,
                                     const int32_t* draft_tokens, const int32_t* parent, const float* u_accept,
                                     const float* u_bonus, float temperature, const tsv_walk_options* opts, int B,
                                     int N, int V, int32_t* accepted_nodes, int32_t* accept_len,
                                     int32_t* bonus_token, int32_t* out_tokens, int32_t* seq_err, void* stream) {
    tsv::SampleArgs a;
    const tsv_status st = reject_args(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus, temperature,
                                      B, N, V, accepted_nodes, accept_len, bonus_token, out_tokens, seq_err, opts, &a);
    if (st != TSV_OK || B == 0) return st;
    cudaError_t e = tsv::launch_tree_reject(a, B, device_sms(), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tree_reject_sample launch");
    return TSV_OK;
}

tsv_status tsv_tree_reject_sample(const float* target_logits, const float* draft_probs,
                                  const int32_t* draft_tokens, const int32_t* parent, const float* u_accept,
                                  const float* u_bonus, float temperature, int B, int N, int V,
                                  int32_t* accepted_nodes, int32_t* accept_len, int32_t* bonus_token,
                                  int32_t* out_tokens, int32_t* seq_err, void* stream) {
    return tsv_tree_reject_sample_ex(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus, temperature,
                                     nullptr, B, N, V, accepted_nodes, accept_len, bonus_token, out_tokens, seq_err,
                                     stream);
}

tsv_status tsv_tree_reject_sample_compact(const float* target_logits, const float* draft_probs,
                                          const int32_t* draft_tokens, const int32_t* parent, const float* u_accept,
                                          const float* u_bonus, float temperature, int B, int N, int V,
                                          int32_t* accepted_nodes, int32_t* accept_len, int32_t* bonus_token,
                                          int32_t* out_tokens, int32_t* seq_err, void* k_cache, void* v_cache,
                                          const int32_t* block_table, const int32_t* seq_lens,
                                          int32_t* new_seq_lens, int Hkv, int D, int block_size, int max_blocks,
                                          int num_blocks, tsv_dtype dtype, int32_t* compact_err, void* stream) {
    return tsv_tree_reject_sample_compact_ex(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus,
                                             temperature, nullptr, B, N, V, accepted_nodes, accept_len, bonus_token,
                                             out_tokens, seq_err, k_cache, v_cache, block_table, seq_lens,
                                             new_seq_lens, Hkv, D, block_size, max_blocks, num_blocks, dtype,
                                             compact_err, stream);
}

tsv_status tsv_tree_reject_sample_compact_ex(const void* target_logits, const float* draft_probs,
                                             const int32_t* draft_tokens, const int32_t* parent,
                                             const float* u_accept, const float* u_bonus, float temperature,
                                             const tsv_walk_options* opts, int B, int N, int V,
                                             int32_t* accepted_nodes, int32_t* accept_len, int32_t* bonus_token,
                                             int32_t* out_tokens, int32_t* seq_err, void* k_cache, void* v_cache,
                                             const int32_t* block_table, const int32_t* seq_lens,
                                             int32_t* new_seq_lens, int Hkv, int D, int block_size, int max_blocks,
                                             int num_blocks, tsv_dtype dtype, int32_t* compact_err, void* stream) {
    tsv::SampleArgs a;
    tsv_status st = reject_args(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus, temperature, B,
                                N, V, accepted_nodes, accept_len, bonus_token, out_tokens, seq_err, opts, &a);
    if (st != TSV_OK) return st;
    st = compact_args(k_cache, v_cache, block_table, seq_lens, new_seq_lens, B, N, Hkv, D, block_size, max_blocks,
                      num_blocks, dtype, compact_err);
    if (st != TSV_OK || B == 0) return st;
    a.k_cache = static_cast<uint8_t*>(k_cache);
    a.v_cache = static_cast<uint8_t*>(v_cache);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.new_seq_lens = new_seq_lens;
    a.compact_err = compact_err;
    a.row_bytes = Hkv * D * (dtype == TSV_F32 ? 4 : 2);
    a.bs_log2 = log2i(block_size);
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    cudaError_t e = tsv::launch_tree_reject(a, B, device_sms(), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tree_reject_sample_compact launch");
    return TSV_OK;
}

tsv_status tsv_kv_compact_accepted(void* k_cache, void* v_cache, const int32_t* block_table,
                                   const int32_t* seq_lens, const int32_t* accepted_nodes,
                                   const int32_t* accept_len, int32_t* new_seq_lens, int B, int N, int Hkv, int D,
                                   int block_size, int max_blocks, int num_blocks, tsv_dtype dtype,
                                   int32_t* seq_err, void* stream) {
    tsv_status st = compact_args(k_cache, v_cache, block_table, seq_lens, new_seq_lens, B, N, Hkv, D, block_size,
                                 max_blocks, num_blocks, dtype, seq_err);
    if (st != TSV_OK || B == 0) return st;
    if (!accepted_nodes || !accept_len) return fail(TSV_ERR_ARG, "null array argument");
    cudaError_t e = tsv::launch_kv_compact(k_cache, v_cache, block_table, seq_lens, accepted_nodes, accept_len,
                                           new_seq_lens, B, N, Hkv, D, block_size, max_blocks, num_blocks,
                                           dtype == TSV_F32 ? 4 : 2, seq_err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_compact_accepted launch");
    return TSV_OK;
}

}  // extern "C"
