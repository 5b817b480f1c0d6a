// attn_common.cuh -- launch plans and shared arguments of the tree-attention kernels.
//
// The rows of a (sequence b, kv head g) pair are the R = N * Gq query rows (node n,
// head h = g*Gq + j) ordered n-major, so one GQA group shares every K/V tile it
// loads; a row group holds up to rows_per_cta of them.
//
// fp32 FMA path (make_attn_plan): one work item = (b, g, key chunk c, row group).
// The prefix of sequence b is cut into nchunks(b) = max(1, ceil(L_b / chunk)) key
// chunks; the last chunk also carries the N tree keys.  A sequence with one chunk
// writes its output directly; otherwise each chunk writes (m, l, O/l) partials to the
// workspace and the merge kernel combines them (log-sum-exp), one warp per row.
//
// bf16 tensor-core path (make_attn_plan_tc): persistent CTAs, `lanes` per row group.
// The keys [0, L_b + N) of every (b, g) unit are cut into 128-key tiles; all units'
// tiles, b-major, form one sequence that is split evenly between the lanes, so every
// CTA streams the same number of K/V tiles whatever the mix of lengths.  A unit that
// straddles lanes leaves (m, l, O/l) partials in per-CTA slots, and a merge kernel over
// all SMs combines them.
#pragma once

#include <cstddef>
#include <cstdint>

namespace tsv {

struct AttnPlan {
    int G;             // query heads per kv head
    int R;             // query rows per (b, kv head) = N * G
    int rows_per_cta;  // rows one work item covers
    int n_rgroups;     // ceil(R / rows_per_cta)
    int chunk;         // prefix keys per chunk (multiple of 128)
    int max_chunks;    // upper bound of nchunks(b) from the block-table capacity
    size_t ws_bytes;   // partials workspace (0 when max_chunks == 1)
    int lanes;         // tensor-core path: persistent CTAs per row group
    int rows_item;     // tensor-core path: rows of a partial slot, min(R, rows_per_cta)
};

// Deterministic function of the shapes and the SM count (the workspace size query
// and the call must agree).
inline AttnPlan make_attn_plan(int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                               int rows_per_cta, int num_sms, int target_waves, int min_chunk) {
    AttnPlan p{};
    p.G = Hq / Hkv;
    p.R = N * p.G;
    p.rows_per_cta = rows_per_cta;
    p.n_rgroups = (p.R + rows_per_cta - 1) / rows_per_cta;
    long long lmax = (long long)max_blocks * block_size - N;  // longest prefix the table can hold
    if (lmax < 0) lmax = 0;
    const long long units = (long long)B * Hkv * p.n_rgroups;
    const long long target = (long long)num_sms * target_waves;
    int chunk = 4096;
    while (chunk > min_chunk && units * ((lmax + chunk - 1) / chunk) < target) chunk >>= 1;
    p.chunk = chunk;
    long long mc = (lmax + chunk - 1) / chunk;
    p.max_chunks = (int)(mc < 1 ? 1 : mc);
    if (p.max_chunks == 1) {
        p.ws_bytes = 0;
    } else {
        const size_t rows = (size_t)B * Hkv * p.max_chunks * p.R;
        p.ws_bytes = rows * (size_t)D * sizeof(float) + 2 * rows * sizeof(float);
    }
    return p;
}

// Tensor-core plan: one CTA per SM (as many lanes as fit beside the row groups), but
// no fewer than about four tiles per CTA at the block table's capacity.  Workspace:
// two partial slots per CTA (its first and its last unit may be pieces), then one
// record per (b, g, row group) unit naming the lanes that hold its pieces.
constexpr int kUnitInfoInts = 8;
inline AttnPlan make_attn_plan_tc(int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                                  int rows_per_cta, int num_sms) {
    AttnPlan p{};
    p.G = Hq / Hkv;
    p.R = N * p.G;
    p.rows_per_cta = rows_per_cta;
    p.n_rgroups = (p.R + rows_per_cta - 1) / rows_per_cta;
    p.rows_item = p.R < rows_per_cta ? p.R : rows_per_cta;
    const long long tiles_cap = (long long)B * Hkv * (((long long)max_blocks * block_size + 127) / 128);
    long long lanes = num_sms / p.n_rgroups;
    if (lanes < 1) lanes = 1;
    if (lanes > (tiles_cap + 3) / 4) lanes = (tiles_cap + 3) / 4;
    if (lanes < 1) lanes = 1;
    p.lanes = (int)lanes;
    p.chunk = 0;
    p.max_chunks = 0;
    const size_t slots = 2 * (size_t)p.lanes * p.n_rgroups;
    p.ws_bytes = slots * p.rows_item * ((size_t)D + 2) * sizeof(float) +
                 (size_t)B * Hkv * p.n_rgroups * kUnitInfoInts * sizeof(int);
    return p;
}

struct AttnArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    // fused append: the tree's K/V rows [B, N, Hkv, D] written into the caches (at
    // logical slots L_b .. L_b + N - 1) before they are read; k_new == nullptr: none
    const void* k_new;
    const void* v_new;
    void* k_cache_w;
    void* v_cache_w;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* parent;
    void* out;
    float* part_o;  // [B][Hkv][max_chunks][R][D]
    float* part_m;  // [B][Hkv][max_chunks][R]
    float* part_l;  // [B][Hkv][max_chunks][R]
    // tensor-core path: part_o [2 * CTAs][rows_item][D], part_m / part_l [2 * CTAs][rows_item]
    int* unit_info;  // [B][Hkv][n_rgroups][8]: first lane, last lane, side of the first piece, -, T (int64)
    int lanes, rows_item;
    int32_t* seq_err;
    int B, N, Hq, Hkv, D;
    int bs_log2, max_blocks, num_blocks;
    float scale_log2;  // scale * log2(e)
    int G, R, rows_per_cta, n_rgroups, chunk, max_chunks;
};

__host__ __device__ inline int num_chunks(int L, int chunk) {
    return L <= 0 ? 1 : (L + chunk - 1) / chunk;
}

}  // namespace tsv
