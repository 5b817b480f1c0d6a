/*
 * tsv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of the target-side verification
 * step of tree-based speculative decoding, written to check the CUDA library
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it; the library never does, and this file shares no code with it.
 *
 * Floating point is accumulated in double (fp64).  Every loop follows the
 * definition of the step directly: no tiling, no online softmax, no split.
 *
 * Sources (pages on tree speculative decoding):
 *  - "Speculative decoding on sglang" (carpedm30 report), sections "What is
 *    Tree-Attention?" and "Tree-based Speculative Decoding (EAGLE) Implementation
 *    Summary": draft candidates are flattened to 1-D and verified in one pass
 *    under a tree mask; the KV cache is updated selectively for accepted indices.
 *  - statistical-learning-notes ch.07 "Speculative Decoding", section "Draft Token
 *    Validation": accept when p >= q, else accept with probability p/q against a
 *    uniform r; on rejection sample from normalize(max(0, p - q)); a fully
 *    accepted run takes one more token from the next-token distribution.
 *  - "Sequoia: Scalable and Robust Speculative Decoding" summary, sections
 *    "Scalable Speculative Decoding" and "Robust Sampling": siblings are verified
 *    as sampling without replacement; its figure comparing the rejection rates of
 *    the SEQUOIA, SpecInfer, SpecTr and top-k verification algorithms: the
 *    SpecInfer variant, read here as siblings drafted independently (with
 *    replacement) from q and verified with the residual update alone, q kept
 *    (with_replacement = 1).
 *  - SGLang "SpeculativeDecoding" page, section "Speculative Decoding" (full /
 *    no / prefix match; rejected tokens' KV cache is evicted).
 *
 * Readings where the pages leave a detail open (each mirrored in the library's
 * header):
 *  - node 0 is the root (the last accepted token, parent -1); its own K/V sits at
 *    tree slot L_b and it is never tested, only its children are;
 *  - a node's ancestor set includes the node itself (a chain then equals causal
 *    attention);
 *  - the distributions used to test node i's children are node i's rows of the
 *    target logits (p = softmax(logits / T)) and of the draft probabilities (q);
 *  - accept iff u < p(x)/q(x) with u in [0,1); q(x) == 0 accepts iff p(x) > 0;
 *  - after a rejected sibling with token x: p <- normalize(max(0, p - q)) (if that
 *    sum is zero, p is kept), q(x) <- 0 and q <- normalize(q) (if that sum is zero,
 *    q is kept), then the next sibling is tried (with replacement: q is kept);
 *  - the bonus token is the smallest t with u_bonus < sum_{v<=t} p(v) (inverse CDF
 *    in token order); if there is none, the last t with p(t) > 0;
 *  - top_k / top_p (the Sequoia summary's table of robustness to top-p; the library
 *    does not offer them yet): p is first filtered to its top_k most probable tokens
 *    and then to the smallest prefix of them, by decreasing p with ties to the lower
 *    index, whose mass reaches top_p, and renormalised; q is the drafter's own
 *    (already filtered) distribution as given;
 *  - at T == 0 a child is accepted iff its token is the argmax of the logits row
 *    (lowest index on ties), and the bonus is that argmax;
 *  - compaction copies the path's K/V rows to contiguous slots after the root and
 *    sets new_seq_len = L_b + 1 + accept_len; eviction is the length cut.
 *
 * Error bits (per sequence, OR-ed): 1 bad tree/path, 2 block id out of range,
 * 4 capacity (L_b + N > max_blocks * block_size, or L_b < 0), 8 token out of range,
 * 16 non-finite logits/probabilities (a visited logits row; the drafted token's
 * draft probability; a node's whole draft row once a residual is formed there).
 * A failed sequence gets accept_len = -1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ORACLE_MUTANT (default 0) plants one known mistake; the pin tests build the
 * mutants to show that each pin fails on them.  The shipped oracle has 0. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ERR_PARENT = 1, ERR_BLOCK = 2, ERR_CAPACITY = 4, ERR_TOKEN = 8, ERR_NONFINITE = 16 };
enum { DT_BF16 = 0, DT_F32 = 1 };

/* ------------------------------------------------------------------ helpers */

static double load_elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == DT_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* parent[0] == -1 and 0 <= parent[i] < i for every other node */
static int tree_is_valid(const int32_t *par, int N)
{
    if (N < 1 || par[0] != -1)
        return 0;
    for (int i = 1; i < N; i++)
        if (par[i] < 0 || par[i] >= i)
            return 0;
    return 1;
}

/* checks capacity and every block id covering logical slots [0, L + N) */
static int cache_errors(const int32_t *bt_row, int L, int N, int bs, int max_blocks, int num_blocks)
{
    if (L < 0 || (int64_t)L + N > (int64_t)max_blocks * bs)
        return ERR_CAPACITY;
    int nblk = (L + N + bs - 1) / bs;
    for (int j = 0; j < nblk; j++)
        if (bt_row[j] < 0 || bt_row[j] >= num_blocks)
            return ERR_BLOCK;
    return 0;
}

/* element index of (logical slot t, kv head h, dim 0) in a [num_blocks, bs, Hkv, D] cache */
static int64_t cache_index(const int32_t *bt_row, int t, int h, int bs, int Hkv, int D)
{
    int64_t phys = (int64_t)bt_row[t / bs] * bs + (t % bs);
    return (phys * Hkv + h) * D;
}

/* ------------------------------------------------------------------ attention */

/*
 * Tree-masked attention.  For query row (b, n, h): the key set is the cached
 * prefix slots 0..L_b-1 plus the tree slots L_b + j for every j on the path from
 * the root to n (n included).  kv head = h / (Hq / Hkv).
 *     s(t) = scale * sum_d q[b,n,h,d] * k[t,d]
 *     w(t) = exp(s(t) - max s) / sum_t' exp(s(t') - max s)
 *     out[d] = sum_t w(t) * v[t,d]
 * rows: flattened (b*N + n)*Hq + h ids to evaluate (NULL = all, in order).
 * out: [nrows][D] doubles.  Rows of a failed sequence are NaN.
 */
int oracle_tree_verify_attn(const void *q, const void *k_cache, const void *v_cache, int dtype,
                            const int32_t *block_table, const int32_t *seq_lens, const int32_t *parent,
                            int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                            int num_blocks, double scale, const int64_t *rows, int64_t nrows,
                            double *out, int32_t *seq_err)
{
    if (B < 0 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || block_size < 1)
        return -1;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; b++) {
        int e = 0;
        if (!tree_is_valid(parent + (int64_t)b * N, N))
            e |= ERR_PARENT;
        e |= cache_errors(block_table + (int64_t)b * max_blocks, seq_lens[b], N, block_size,
                          max_blocks, num_blocks);
        seq_err[b] = e;
    }
    int max_keys = 0;
    for (int b = 0; b < B; b++)
        if (seq_lens[b] + N > max_keys)
            max_keys = seq_lens[b] + N;
    int *keys = malloc(sizeof(int) * (size_t)(max_keys > 0 ? max_keys : 1));
    double *s = malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    unsigned char *on_path = malloc((size_t)N);
    int64_t total = rows ? nrows : (int64_t)B * N * Hq;

    for (int64_t r = 0; r < total; r++) {
        int64_t id = rows ? rows[r] : r;
        int h = (int)(id % Hq);
        int n = (int)((id / Hq) % N);
        int b = (int)(id / ((int64_t)Hq * N));
        double *o = out + r * D;
        if (seq_err[b]) {
            for (int d = 0; d < D; d++)
                o[d] = NAN;
            continue;
        }
        const int32_t *par = parent + (int64_t)b * N;
        const int32_t *bt = block_table + (int64_t)b * max_blocks;
        const int L = seq_lens[b];
#if ORACLE_MUTANT == 4
        const int kvh = h % Hkv; /* mistake: interleaved instead of grouped heads */
#else
        const int kvh = h / G;
#endif

        /* key set: the whole prefix, then the root-to-n path in tree order */
        memset(on_path, 0, (size_t)N);
        for (int a = n; a >= 0; a = par[a])
            on_path[a] = 1;
#if ORACLE_MUTANT == 3
        on_path[n] = (n == 0); /* mistake: a node does not see itself */
#endif
        int nk = 0;
        for (int t = 0; t < L; t++)
            keys[nk++] = t;
        for (int j = 0; j < N; j++)
            if (on_path[j])
                keys[nk++] = L + j;

        const int64_t qoff = id * D;
        double mx = -INFINITY;
        for (int i = 0; i < nk; i++) {
            int64_t koff = cache_index(bt, keys[i], kvh, block_size, Hkv, D);
            double acc = 0.0;
            for (int d = 0; d < D; d++)
                acc += load_elem(q, dtype, qoff + d) * load_elem(k_cache, dtype, koff + d);
            s[i] = scale * acc;
            if (s[i] > mx)
                mx = s[i];
        }
        double z = 0.0;
        for (int i = 0; i < nk; i++) {
            s[i] = exp(s[i] - mx);
            z += s[i];
        }
        for (int d = 0; d < D; d++)
            o[d] = 0.0;
        for (int i = 0; i < nk; i++) {
            int64_t voff = cache_index(bt, keys[i], kvh, block_size, Hkv, D);
            double w = s[i] / z;
            for (int d = 0; d < D; d++)
                o[d] += w * load_elem(v_cache, dtype, voff + d);
        }
    }
    free(keys);
    free(s);
    free(on_path);
    return 0;
}

/* ------------------------------------------------------------------ verifier */

static int argmax_row(const float *row, int V)
{
    int best = 0;
    for (int v = 1; v < V; v++)
        if (row[v] > row[best])
            best = v;
    return best;
}

static int row_is_finite(const float *row, int V)
{
    for (int v = 0; v < V; v++)
        if (!isfinite(row[v]))
            return 0;
    return 1;
}

/* Filtered target distribution (top-k / top-p): keep the top_k most probable tokens
 * (top_k <= 0: all), then the smallest prefix of them, in order of decreasing p (ties:
 * lower index first), whose mass reaches top_p of the row (top_p >= 1: all kept); zero
 * the rest and renormalise.  tmp holds V (p, index) pairs. */
typedef struct {
    double p;
    int v;
} pv_t;

static int pv_cmp(const void *a, const void *b)
{
    const pv_t *x = (const pv_t *)a, *y = (const pv_t *)b;
    if (x->p != y->p)
        return x->p > y->p ? -1 : 1;
    return x->v - y->v;
}

static void filter_top(double *p, int V, int top_k, double top_p, pv_t *tmp)
{
    if (top_k <= 0 && top_p >= 1.0)
        return;
    for (int v = 0; v < V; v++) {
        tmp[v].p = p[v];
        tmp[v].v = v;
    }
    qsort(tmp, (size_t)V, sizeof(pv_t), pv_cmp);
    int keep = (top_k > 0 && top_k < V) ? top_k : V;
    if (top_p < 1.0) {
        double cum = 0.0;
        int n = 0;
        while (n < keep) {
            cum += tmp[n].p;
            n++;
            if (cum >= top_p)
                break;
        }
        keep = n;
    }
    for (int v = 0; v < V; v++)
        p[v] = 0.0;
    double z = 0.0;
    for (int n = 0; n < keep; n++)
        z += tmp[n].p;
    for (int n = 0; n < keep; n++)
        p[tmp[n].v] = tmp[n].p / z;
}

/*
 * Rejection-sampling tree walk (one sequence after another).  target_logits is
 * float32 (logits_dtype = DT_F32) or bfloat16 bits (DT_BF16).
 *
 * Outputs per sequence b: accepted_nodes[b, 0..] = root-first path (-1 padded),
 * accept_len[b] = drafts accepted (path length - 1), bonus_token[b], and
 * out_tokens[b, 0..] = accepted draft tokens followed by the bonus (-1 padded).
 *
 * Optional records for the parity tests: ratio[b, c] = p(x)/q(x) for every child c
 * that was tried (NaN otherwise; +inf when q(x) == 0 < p(x)); bonus_cdf[b] =
 * (sum_{v<t} p(v), sum_{v<=t} p(v)) around the bonus token t (T > 0 only).
 */
int oracle_tree_reject_sample(const void *target_logits, const float *draft_probs,
                              const int32_t *draft_tokens, const int32_t *parent,
                              const float *u_accept, const float *u_bonus, float temperature,
                              int B, int N, int V, int32_t *accepted_nodes, int32_t *accept_len,
                              int32_t *bonus_token, int32_t *out_tokens, double *ratio,
                              double *bonus_cdf, int32_t *seq_err, int with_replacement, int top_k,
                              double top_p, int logits_dtype)
{
    if (B < 0 || N < 1 || V < 1 || !(temperature >= 0.0f) || !isfinite(temperature))
        return -1;
    const int greedy = (temperature == 0.0f);
    const double T = (double)temperature;
    double *p = malloc(sizeof(double) * (size_t)V);
    float *rowbuf = malloc(sizeof(float) * (size_t)V); /* the visited logits row, decoded */
    double *qv = malloc(sizeof(double) * (size_t)V);
    int32_t *path = malloc(sizeof(int32_t) * (size_t)N);
    pv_t *pv = (top_k > 0 || top_p < 1.0) ? malloc(sizeof(pv_t) * (size_t)V) : NULL;

    for (int b = 0; b < B; b++) {
        const int32_t *par = parent + (int64_t)b * N;
        const int32_t *tok = draft_tokens + (int64_t)b * N;
        int32_t *acc_row = accepted_nodes + (int64_t)b * N;
        int32_t *out_row = out_tokens + (int64_t)b * N;
        for (int j = 0; j < N; j++) {
            acc_row[j] = -1;
            out_row[j] = -1;
            if (ratio)
                ratio[(int64_t)b * N + j] = NAN;
        }
        if (bonus_cdf) {
            bonus_cdf[2 * b] = NAN;
            bonus_cdf[2 * b + 1] = NAN;
        }
        accept_len[b] = -1;
        bonus_token[b] = -1;
        seq_err[b] = 0;
        if (!tree_is_valid(par, N)) {
            seq_err[b] = ERR_PARENT;
            continue;
        }

        int err = 0;
        int plen = 0;
        int i = 0;
        path[plen++] = 0;
        const float *row = NULL;
        for (;;) {
            /* bf16 logits decode exactly to float (the 16 bits are the top of a float) */
            for (int v = 0; v < V; v++)
#if ORACLE_MUTANT == 7 /* mistake: bf16 bits converted as an integer value, not reinterpreted */
                rowbuf[v] = logits_dtype == DT_F32
                                ? ((const float *)target_logits)[((int64_t)b * N + i) * V + v]
                                : (float)((const uint16_t *)target_logits)[((int64_t)b * N + i) * V + v];
#else
                rowbuf[v] = (float)load_elem(target_logits, logits_dtype, ((int64_t)b * N + i) * V + v);
#endif
            row = rowbuf;
            if (!row_is_finite(row, V)) {
                err = ERR_NONFINITE;
                break;
            }
            int amax = argmax_row(row, V);
            int q_loaded = 0;
            if (!greedy) {
                /* p = softmax(logits_i / T) */
                double mx = (double)row[amax];
                double z = 0.0;
                for (int v = 0; v < V; v++) {
                    p[v] = exp(((double)row[v] - mx) / T);
                    z += p[v];
                }
                for (int v = 0; v < V; v++)
                    p[v] /= z;
                filter_top(p, V, top_k, top_p, pv);
            }
            const float *qrow = draft_probs ? draft_probs + ((int64_t)b * N + i) * V : NULL;
            int next = -1;
            for (int c = i + 1; c < N && !err; c++) {
                if (par[c] != i)
                    continue;
                int x = tok[c];
                if (x < 0 || x >= V) {
                    err = ERR_TOKEN;
                    break;
                }
                if (greedy) {
                    if (x == amax) {
                        next = c;
                        break;
                    }
                    continue;
                }
                /* q(x): node i's draft probability of the drafted token; the whole
                 * row is read only once a residual has to be formed */
                double qx;
                if (q_loaded) {
                    qx = qv[x];
                } else {
                    if (!isfinite(qrow[x])) {
                        err = ERR_NONFINITE;
                        break;
                    }
                    qx = (double)qrow[x];
                }
                double r;
                if (qx > 0.0)
                    r = p[x] / qx;
                else
                    r = (p[x] > 0.0) ? INFINITY : 0.0;
                if (ratio)
                    ratio[(int64_t)b * N + c] = r;
                if ((double)u_accept[(int64_t)b * N + c] < r) {
                    next = c;
                    break;
                }
                if (!q_loaded) {
                    if (!row_is_finite(qrow, V)) {
                        err = ERR_NONFINITE;
                        break;
                    }
                    for (int v = 0; v < V; v++)
                        qv[v] = (double)qrow[v];
                    q_loaded = 1;
                }
                /* rejected: residual p <- normalize(max(0, p - q)) */
                double zr = 0.0;
                for (int v = 0; v < V; v++)
                    zr += fmax(0.0, p[v] - qv[v]);
#if ORACLE_MUTANT == 2
                zr = 1.0; /* mistake: residual left unnormalised */
#endif
#if ORACLE_MUTANT != 5
                if (zr > 0.0)
                    for (int v = 0; v < V; v++)
                        p[v] = fmax(0.0, p[v] - qv[v]) / zr;
#endif
                /* without replacement: q(x) <- 0, q <- normalize(q); with replacement
                 * the next sibling was drawn from the same q, which is kept */
                if (!with_replacement) {
                    qv[x] = 0.0;
                    double zq = 0.0;
                    for (int v = 0; v < V; v++)
                        zq += qv[v];
                    if (zq > 0.0)
                        for (int v = 0; v < V; v++)
                            qv[v] /= zq;
                }
            }
            if (err || next < 0)
                break;
            path[plen++] = next;
            i = next;
        }
        if (err) {
            seq_err[b] = err;
            for (int j = 0; j < N; j++)
                if (ratio)
                    ratio[(int64_t)b * N + j] = NAN;
            continue;
        }

        /* bonus token from the final node */
        int bonus;
        if (greedy) {
            bonus = argmax_row(row, V);
        } else {
            double u = (double)u_bonus[b];
            double cum = 0.0, lo = 0.0;
            bonus = -1;
            for (int v = 0; v < V; v++) {
                lo = cum;
                cum += p[v];
                if (u < cum) {
                    bonus = v;
                    break;
                }
            }
            if (bonus < 0) {
                for (int v = V - 1; v >= 0; v--)
                    if (p[v] > 0.0) {
                        bonus = v;
                        break;
                    }
                cum = 0.0;
                for (int v = 0; v <= bonus; v++) {
                    lo = cum;
                    cum += p[v];
                }
            }
            if (bonus_cdf) {
                bonus_cdf[2 * b] = lo;
                bonus_cdf[2 * b + 1] = cum;
            }
        }
        for (int j = 0; j < plen; j++)
            acc_row[j] = path[j];
        for (int j = 1; j < plen; j++)
            out_row[j - 1] = tok[path[j]];
        out_row[plen - 1] = bonus;
        accept_len[b] = plen - 1;
        bonus_token[b] = bonus;
    }
    free(p);
    free(rowbuf);
    free(qv);
    free(pv);
    free(path);
    return 0;
}

/* ------------------------------------------------------------------ compaction */

/*
 * KV-cache rewrite for the accepted path: for j = 1..accept_len the K and V rows of
 * logical slot L_b + accepted_nodes[b, j] (all kv heads) are copied to logical slot
 * L_b + j, and new_seq_lens[b] = L_b + 1 + accept_len[b].  Slots at or beyond the new
 * length are evicted (left as they are; the length cut frees them).  Every path
 * row is gathered into a temporary buffer before any is written.
 * A sequence with accept_len < 0 is left untouched (new length = L_b).
 */
int oracle_kv_compact_accepted(void *k_cache, void *v_cache, int dtype, const int32_t *block_table,
                               const int32_t *seq_lens, const int32_t *accepted_nodes,
                               const int32_t *accept_len, int32_t *new_seq_lens, int B, int N,
                               int Hkv, int D, int block_size, int max_blocks, int num_blocks,
                               int32_t *seq_err)
{
    if (B < 0 || N < 1 || Hkv < 1 || D < 1 || block_size < 1)
        return -1;
    const size_t esz = dtype == DT_F32 ? 4 : 2;
    const size_t row_bytes = (size_t)Hkv * D * esz;
    unsigned char *tmp = malloc(2 * row_bytes * (size_t)N);
    for (int b = 0; b < B; b++) {
        const int L = seq_lens[b];
        const int A = accept_len[b];
        const int32_t *path = accepted_nodes + (int64_t)b * N;
        const int32_t *bt = block_table + (int64_t)b * max_blocks;
        seq_err[b] = 0;
        new_seq_lens[b] = L;
        if (A < 0)
            continue;
        int e = 0;
        if (A > N - 1 || path[0] != 0)
            e |= ERR_PARENT;
        for (int j = 1; j <= A && !e; j++)
            if (path[j] <= path[j - 1] || path[j] >= N)
                e |= ERR_PARENT;
        if (!e)
            e |= cache_errors(bt, L, N, block_size, max_blocks, num_blocks);
        if (e) {
            seq_err[b] = e;
            continue;
        }
        /* gather */
        for (int j = 1; j <= A; j++) {
            int64_t src = cache_index(bt, L + path[j], 0, block_size, Hkv, D);
            memcpy(tmp + (size_t)(j - 1) * 2 * row_bytes, (unsigned char *)k_cache + src * esz, row_bytes);
            memcpy(tmp + (size_t)(j - 1) * 2 * row_bytes + row_bytes, (unsigned char *)v_cache + src * esz,
                   row_bytes);
        }
        /* scatter to contiguous slots after the root */
        for (int j = 1; j <= A; j++) {
#if ORACLE_MUTANT == 6
            int64_t dst = cache_index(bt, L + j - 1, 0, block_size, Hkv, D); /* mistake: off by one */
#else
            int64_t dst = cache_index(bt, L + j, 0, block_size, Hkv, D);
#endif
            memcpy((unsigned char *)k_cache + dst * esz, tmp + (size_t)(j - 1) * 2 * row_bytes, row_bytes);
            memcpy((unsigned char *)v_cache + dst * esz, tmp + (size_t)(j - 1) * 2 * row_bytes + row_bytes,
                   row_bytes);
        }
        new_seq_lens[b] = L + 1 + A;
    }
    free(tmp);
    return 0;
}
