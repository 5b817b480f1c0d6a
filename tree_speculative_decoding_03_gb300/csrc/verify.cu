// verify.cu -- rejection-sampling walk of the draft tree, one thread-block cluster
// per sequence.
//
// statistical-learning-notes ch.07 "Speculative Decoding", section "Draft Token
// Validation": accept x when p(x) >= q(x), else with probability p(x)/q(x); on a
// rejection the next token comes from normalize(max(0, p - q)); a fully accepted
// run takes one more token from the next-token distribution.  Sequoia summary,
// sections "Scalable Speculative Decoding" / "Robust Sampling": siblings are
// verified as sampling without replacement (after a rejected sibling x, q(x) <- 0
// and q is renormalised before the next sibling is tried).
//
// Design (GB300): the walk is sequential, so its cost is the latency of one
// vocabulary-wide pass per visited node.  The vocabulary row is split over the
// CTAs of a cluster (up to 16) and over their threads; every thread keeps its
// slice of the current node's logits (and, after a rejection, draft probabilities)
// in registers, loaded with coalesced 128-bit loads.  Reductions go warp shuffles
// (fp32) -> one warp per CTA -> DSMEM across the cluster; every CTA combines the
// cluster partials in the same order, so all CTAs hold bit-identical scalars and
// take identical decisions without a second exchange.  The first child's logits
// row is prefetched into L2 while the current row is reduced, and the children's
// scalars are copied asynchronously (cp.async) while it is reduced.
//
// Precision without fp64: GB300's fp64 rate is a small fraction of fp32, so sums
// across threads, warps and CTAs are carried as float-float pairs (error-free
// two-sum/two-product transformations, about 44 significant bits), and the
// acceptance ratio p(x)/q(x) is formed in float-float from a compensated exponent
// argument; its error is dominated by expf's (<= 2 ulp), a few 1e-7 relative.
// Vocabulary-wide passes take each entry as 2^(l c - MC) with c = log2(e) / T and
// MC = fl(M c) (one FMA and one ex2.approx, ~2 ulp): the same offset for every entry
// keeps the pass's p self-normalised, and the normaliser handed to the ratio is
// corrected by the exactly computed rounding of M c.
//
// The children of the current node are tested in parallel lanes: each keeps its
// (p(x), q(x)) at the current residual level in shared memory, updated once per
// rejection, so a test is a comparison and a rejection costs one pass and one
// cluster reduction whatever the number of earlier rejections.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <map>
#include <mutex>

#include "compact_path.cuh"
#include "verify_args.cuh"

namespace cg = cooperative_groups;

namespace tsv {

constexpr int kMaxRejections = kMaxNodes;  // at most one per tried child

// ----------------------------------------------------------------------------- float-float

struct ff {
    float hi, lo;
};
__device__ __forceinline__ ff ff_make(float a) { return ff{a, 0.0f}; }
// a + b exactly as hi + lo (Knuth's two-sum)
__device__ __forceinline__ ff two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    const float e = (a - (s - bb)) + (b - bb);
    return ff{s, e};
}
// the same when |a| >= |b| (Dekker's fast two-sum)
__device__ __forceinline__ ff quick_two_sum(float a, float b) {
    const float s = a + b;
    return ff{s, b - (s - a)};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    const ff s = two_sum(a.hi, b.hi);
    return quick_two_sum(s.hi, s.lo + (a.lo + b.lo));
}
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff{-b.hi, -b.lo}); }
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
    const float p = a.hi * b;
    float e = fmaf(a.hi, b, -p);
    e = fmaf(a.lo, b, e);
    return quick_two_sum(p, e);
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
    const float p = a.hi * b.hi;
    float e = fmaf(a.hi, b.hi, -p);
    e = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
    return quick_two_sum(p, e);
}
// 1 / b: a correctly rounded reciprocal of b.hi refined by one float-float step
__device__ __forceinline__ ff ff_recip(ff b) {
    const float q1 = __frcp_rn(b.hi);
    const ff r = ff_sub(ff_make(1.0f), ff_mul_f(b, q1));
    return quick_two_sum(q1, r.hi * q1);
}
__device__ __forceinline__ ff ff_div(ff a, ff b) {
    const float q1 = a.hi / b.hi;
    const ff r = ff_sub(a, ff_mul_f(b, q1));
    const float q2 = r.hi / b.hi;
    return quick_two_sum(q1, q2);
}
__device__ __forceinline__ float ff_float(ff a) { return a.hi + a.lo; }
__device__ __forceinline__ bool ff_pos(ff a) { return a.hi > 0.0f || (a.hi == 0.0f && a.lo > 0.0f); }
__device__ __forceinline__ bool ff_lt(ff a, ff b) { return ff_pos(ff_sub(b, a)); }
__device__ __forceinline__ ff ff_max0(ff a) { return ff_pos(a) ? a : ff_make(0.0f); }

// ----------------------------------------------------------------------------- warp helpers

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ff w{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
        v = ff_add(v, w);
    }
    return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// (value, index) argmax with ties to the lower index
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (v2 > v || (v2 == v && i2 < i)) {
            v = v2;
            i = i2;
        }
    }
}

// ----------------------------------------------------------------------------- async copies
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
// one 4-byte global -> shared copy that completes asynchronously (cp.async.wait_group)
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// true iff v is one of the first j rejected tokens xr[0..j-1]
__device__ __forceinline__ bool is_rejected(int v, int j, const int* xr) {
    for (int i = 0; i < j; ++i)
        if (xr[i] == v) return true;
    return false;
}

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// four consecutive logits starting at a 4-entry boundary: one 16-byte (fp32) or
// 8-byte (bf16) load
__device__ __forceinline__ void load4_aligned(const float* p, float (&x)[4]) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = t.x;
    x[1] = t.y;
    x[2] = t.z;
    x[3] = t.w;
}
__device__ __forceinline__ void load4_aligned(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = __uint_as_float(t.x << 16);  // a bf16 value is the top half of the float
    x[1] = __uint_as_float(t.x & 0xffff0000u);
    x[2] = __uint_as_float(t.y << 16);
    x[3] = __uint_as_float(t.y & 0xffff0000u);
}

template <int VEC, bool ALIGNED, typename TL>
__device__ __forceinline__ void load_slice(const TL* row, int v0, int v1, float (&x)[VEC][4], float fill) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int base = v0 + (k * (int)blockDim.x + (int)threadIdx.x) * 4;
        if (ALIGNED) {
            if (base < v1) {
                load4_aligned(row + base, x[k]);
            } else {
                x[k][0] = x[k][1] = x[k][2] = x[k][3] = fill;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[k][e] = (base + e < v1) ? to_f32(row[base + e]) : fill;
        }
    }
}

// this thread's 4 entries of vector step k (fill past v1)
template <bool ALIGNED>
__device__ __forceinline__ void load4(const float* row, int base, int v1, float (&x)[4], float fill) {
    if (ALIGNED) {
        if (base < v1) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(row + base));
            x[0] = t.x;
            x[1] = t.y;
            x[2] = t.z;
            x[3] = t.w;
        } else {
            x[0] = x[1] = x[2] = x[3] = fill;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = (base + e < v1) ? __ldg(row + base + e) : fill;
    }
}

// Bit (4k + e) set iff this thread's entry e of vector step k is one of the tokens
// xr[0..n-1] (the rejected siblings at the current node): an O(n) scan per pass
// instead of an O(n) membership test per entry.
template <int VEC>
__device__ __forceinline__ uint64_t owned_mask(const int* xr, int n, int v0, int v1) {
    uint64_t m = 0ull;
    for (int i = 0; i < n; ++i) {
        const int x = xr[i];
        if (x < v0 || x >= v1) continue;
        const int f = (x - v0) >> 2;
        if (f % (int)blockDim.x != (int)threadIdx.x) continue;
        const int k = f / (int)blockDim.x;
        if (k < VEC) m |= 1ull << (k * 4 + ((x - v0) & 3));
    }
    return m;
}

template <int VEC, typename TL>
__device__ __forceinline__ void prefetch_slice(const TL* row, int v0, int v1) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int base = v0 + (k * (int)blockDim.x + (int)threadIdx.x) * 4;
        // one prefetch per 128-byte line: the thread whose four entries start the line
        if (base < v1 && ((reinterpret_cast<uintptr_t>(row + base) & 127) < 4 * sizeof(TL))) prefetch_l2(row + base);
    }
}

// One CTA's contribution to a cluster reduction.
struct __align__(16) RedSlot {
    float a;   // max / argmax value
    float hi;  // float-float sum (or second sum's hi in kind 1)
    float lo;
    int i;     // argmax index, or second sum's hi bits
    int flag;  // OR-ed error flag
    float hi2, lo2;
    int pad;
};

enum { kRedStats = 0, kRedSums = 1, kRedArgmax = 2 };
constexpr int kMaxCluster = 16;  // CTAs of a walk's cluster

// Cluster all-reduce: every CTA writes `mine` into slot [parity][its rank] of every CTA
// of the cluster (remote stores, issued before the barrier), the cluster synchronises,
// and warp 0 of every CTA combines its own, now local, slots in rank order (so every
// CTA obtains bit-identical results).  Stats: (raw max a, sum hi+lo of
// 2^(x c - fl(a c))) with per-slot rescaling; sums: two float-float sums; argmax:
// (a, i).  Must be called by every thread of every CTA; the result is in *res
// after the closing __syncthreads.  Slots alternate by parity, so the writes of the
// next reduction cannot overtake a slow CTA still reading this one: they follow the
// next barrier, which the slow CTA passes only after its reads.  slots: [2][kMaxCluster].
struct NoPost {
    __device__ void operator()(const RedSlot&) const {}
};
template <typename Post = NoPost>
__device__ __forceinline__ void cluster_allreduce(cg::cluster_group& cluster, RedSlot* slots, int parity,
                                                  const RedSlot& mine, int kind, float c2, RedSlot* res,
                                                  bool wait_async = false, const Post& post = Post()) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int cs = (int)cluster.num_blocks();
    // `mine` was written by a lane of warp 0 (the callers need no block barrier before the
    // call: the cluster barrier below holds every thread)
    if (tid < 32) __syncwarp();
    if (tid < cs) *cluster.map_shared_rank(&slots[parity * kMaxCluster + cluster.block_rank()], tid) = mine;
    // the last warp's asynchronous copies (issued before the row pass) have landed by the
    // cluster barrier, which makes them visible to warp 0's post-step
    if (wait_async && (tid >> 5) == (int)(blockDim.x >> 5) - 1) asm volatile("cp.async.wait_all;" ::: "memory");
    cluster.sync();
    if (tid < 32) {
        RedSlot r{};
        r.a = -INFINITY;
        r.i = 0x7fffffff;
        if (lane < cs) r = slots[parity * kMaxCluster + lane];
        const int flag = warp_or(lane < cs ? r.flag : 0);
        RedSlot o{};
        o.flag = flag;
        if (kind == kRedStats) {
            const float m = warp_max(lane < cs ? r.a : -INFINITY);
            ff c = ff_make(0.0f);
            if (lane < cs && (r.hi > 0.0f)) c = ff_mul_f(ff{r.hi, r.lo}, exp2f(r.a * c2 - m * c2));
            c = warp_sum_ff(c);
            o.a = m;
            o.hi = c.hi;
            o.lo = c.lo;
        } else if (kind == kRedSums) {
            ff c1 = lane < cs ? ff{r.hi, r.lo} : ff_make(0.0f);
            ff c2 = lane < cs ? ff{r.hi2, r.lo2} : ff_make(0.0f);
            c1 = warp_sum_ff(c1);
            c2 = warp_sum_ff(c2);
            o.hi = c1.hi;
            o.lo = c1.lo;
            o.hi2 = c2.hi;
            o.lo2 = c2.lo;
        } else {
            float v = lane < cs ? r.a : -INFINITY;
            int i = lane < cs ? r.i : 0x7fffffff;
            warp_argmax(v, i);
            o.a = v;
            o.i = i;
        }
        if (lane == 0) *res = o;
        post(o);  // warp 0, every lane holds the combined result
    }
    __syncthreads();
}

// Recomputes the normalised p of residual level `level` into the register slice from
// the logits row and the recorded levels (the slow, per-entry chain; used only when a
// residual sum is exactly zero).
template <int VEC, bool ALIGNED, typename TL>
__device__ __forceinline__ void rebuild_level(float (&lv)[VEC][4], const TL* lrow, const float* qrow, int v0, int v1,
                                           int level, float c2, float MC, float invZ, const int* xrej,
                                           const float* inv_sq, const float* inv_zr, const int* zr_ok,
                                           bool replacement) {
    load_slice<VEC, ALIGNED>(lrow, v0, v1, lv, -INFINITY);
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int base = v0 + (k * (int)blockDim.x + (int)threadIdx.x) * 4;
        float qk[4];
        load4<ALIGNED>(qrow, base, v1, qk, 0.0f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = base + e;
            float p = ex2(fmaf(lv[k][e], c2, -MC)) * invZ;
            for (int j = 1; j <= level; ++j) {
                const float qprev = (j == 1 || replacement) ? qk[e]
                                                            : (is_rejected(v, j - 1, xrej) ? 0.0f : qk[e] * inv_sq[j - 1]);
                if (zr_ok[j]) p = fmaxf(0.0f, p - qprev) * inv_zr[j];
            }
            lv[k][e] = (v < v1) ? p : 0.0f;
        }
    }
}

// Order key of a logit: a larger float has a larger key (sign-magnitude to biased).
__device__ __forceinline__ uint32_t order_key(float l) {
    const uint32_t u = __float_as_uint(l);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Fused tail (rank 0 of the cluster, every thread): the KV-cache rewrite of the
// accepted path, exactly as the compaction kernel does it; A < 0 (walk error) leaves
// the sequence untouched.
__device__ __forceinline__ void fused_compact(const SampleArgs& a, int b, int A, const int* path, int* s_flag,
                                              int* s_path, int block_err) {
    const int L = a.seq_lens[b];
    int e = 0;
    if (A >= 0)
        e = compact_path(a.k_cache, a.v_cache, a.block_table + (long long)b * a.max_blocks, L, A, path, a.N,
                         a.row_bytes, a.bs_log2, a.max_blocks, a.num_blocks, s_flag, s_path, block_err);
    if (threadIdx.x == 0) {
        a.compact_err[b] = e;
        a.new_seq_lens[b] = (A < 0 || e) ? L : L + 1 + A;
    }
}

template <int VEC, bool ALIGNED, typename TL>
// 16 vector steps per thread run with at most 384 threads (168 registers a thread)
__global__ void __launch_bounds__(VEC > 8 ? 384 : 512, 1) tree_reject_kernel(const SampleArgs a) {
    pdl_wait();  // the inputs may come from the previous kernel in the stream
    pdl_launch_dependents();
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int N = a.N, V = a.V;
    const int v0 = min(V, rank * a.v_per_cta), v1 = min(V, v0 + a.v_per_cta);
    const bool greedy = (a.T == 0.0f);
    const float T = a.T;
    const float c2 = greedy ? 0.0f : 1.4426950408889634f / a.T;  // log2(e) / T

    __shared__ int s_par[kMaxNodes], s_tok[kMaxNodes], s_path[kMaxNodes];
    __shared__ int s_rank[kMaxNodes];  // a child's place among its siblings (set-up only)
    // [node parity][child]: a node's copies start while slower warps may still test the previous node's
    __shared__ float s_lx2[2 * kMaxNodes], s_qx2[2 * kMaxNodes], s_ux2[2 * kMaxNodes];
    // per child of the current node: p(x), q(x) at the current residual level, and
    // whether its token has already been rejected at this node
    __shared__ ff s_px[kMaxNodes], s_qc[kMaxNodes];
    __shared__ int s_rflag[kMaxNodes];
    __shared__ RedSlot s_red[2 * kMaxCluster];  // [parity][source rank]
    __shared__ RedSlot s_cta;  // this CTA's partial
    __shared__ RedSlot s_all;  // cluster result
    __shared__ float s_wf[32], s_wg[32];
    __shared__ int s_wi[32], s_wb[32];
    __shared__ int s_flag;
    // rejection history at the current node
    __shared__ int s_xrej[kMaxRejections];        // rejected tokens x_1..x_j
    __shared__ ff s_zr[kMaxRejections + 1];       // residual sums Zr_j (level j >= 1)
    __shared__ ff s_sq[kMaxRejections + 1];       // S_j = sum of q over tokens not in {x_1..x_j}
    __shared__ float s_inv_zr[kMaxRejections + 1], s_inv_sq[kMaxRejections + 1];
    __shared__ int s_zr_ok[kMaxRejections + 1];
    __shared__ float s_seg[16 * 16];  // bonus: [k][warp] segment sums (VEC <= 16, <= 16 warps)
    __shared__ ff s_segcum[16 * 16];  // bonus: inclusive prefix over (k, warp)
    __shared__ ff s_target;
    __shared__ int s_claim, s_segsel;
    // aligned rows: the first rejection pass at a node keeps this CTA's slice of the
    // node's draft row in shared memory for the node's later passes
    extern __shared__ float4 s_dyn[];
    float* s_q = reinterpret_cast<float*>(s_dyn);
    const bool bulk = ALIGNED && v1 > v0;
    const ff invT_ff = greedy ? ff_make(0.0f) : ff_div(ff_make(1.0f), ff_make(T));
    // top-k / top-p filter of the target at every visited node (0 / 1: none)
    const bool filtered = (a.top_k > 0 && a.top_k < V) || a.top_p < 1.0f;
    const float kt = (a.top_k > 0 && a.top_k < V) ? (float)a.top_k : 3.0e38f;

    int parity = 0;
    // Block then cluster sum of two per-thread fp32 values (float-float across warps and
    // CTAs, combined in rank order): the results are in s_all (hi, lo) and (hi2, lo2).
    // Called by every thread of every CTA.
    auto reduce_sums = [&](float x, float y) {
        x = warp_sum(x);
        y = warp_sum(y);
        if (lane == 0) {
            s_wf[warp] = x;
            s_wg[warp] = y;
        }
        __syncthreads();
        if (warp == 0) {
            const ff z1 = warp_sum_ff(ff_make(lane < nwarps ? s_wf[lane] : 0.0f));
            const ff z2 = warp_sum_ff(ff_make(lane < nwarps ? s_wg[lane] : 0.0f));
            if (lane == 0) {
                RedSlot r{};
                r.hi = z1.hi;
                r.lo = z1.lo;
                r.hi2 = z2.hi;
                r.lo2 = z2.lo;
                s_cta = r;
            }
        }
        cluster_allreduce(cluster, s_red, parity, s_cta, kRedSums, c2, &s_all);
        parity ^= 1;
    };

    // fused rewrite (rank 0): the last warp checks the sequence's cache blocks now, while
    // the walk runs, so the tail only checks the path and moves the rows
    __shared__ int s_blkerr;
    if (a.k_cache != nullptr && rank == 0 && warp == nwarps - 1) {
        const int e = warp_cache_errors(a.block_table + (long long)b * a.max_blocks, a.seq_lens[b], N,
                                        1 << a.bs_log2, a.max_blocks, a.num_blocks);
        if (lane == 0) s_blkerr = e;
    }

    // ---- tree and tokens
    for (int i = tid; i < N; i += blockDim.x) {
        s_par[i] = a.parent[(long long)b * N + i];
        s_tok[i] = a.tokens[(long long)b * N + i];
    }
    const bool tree_ok = block_tree_ok(a.parent + (long long)b * N, N, &s_flag);

    int err = tree_ok ? 0 : TSV_DERR_PARENT;
    int node = 0, plen = 1;
    if (tid == 0) s_path[0] = 0;
    // children of every node in index order, once (warp 0): node i's children are
    // s_kidlist[s_kstart[i] .. s_kstart[i] + s_kcnt[i]).  A child's place among its
    // siblings is its parent's count so far plus its rank among the lanes of its chunk
    // with the same parent.
    __shared__ int s_kcnt[kMaxNodes], s_kstart[kMaxNodes], s_kidlist[kMaxNodes];
    if (tree_ok && warp == 0) {
        for (int i = lane; i < N; i += 32) s_kcnt[i] = 0;
        __syncwarp();
        for (int base = 1; base < N; base += 32) {
            const int c = base + lane;
            const bool has = c < N;
            const int p = has ? s_par[c] : -1 - lane;  // lanes past N: a parent of their own
            const unsigned same = __match_any_sync(0xffffffffu, p);
            const int within = __popc(same & ((1u << lane) - 1u));
            const int before = has ? s_kcnt[p] : 0;
            __syncwarp();
            if (has) {
                s_rank[c] = before + within;
                if (within == 0) s_kcnt[p] = before + __popc(same);
            }
            __syncwarp();
        }
        int carry = 0;  // exclusive prefix of the counts
        for (int base = 0; base < N; base += 32) {
            const int i = base + lane;
            const int v = i < N ? s_kcnt[i] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (i < N) s_kstart[i] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        for (int c = 1 + lane; c < N; c += 32) s_kidlist[s_kstart[s_par[c]] + s_rank[c]] = c;
    }
    __syncthreads();
    // the current node's logits slice stays in registers; its draft row is re-read (from
    // L2, where it was prefetched) by the passes that need it, which keeps register
    // pressure low enough for 32 entries per thread
    float lv[VEC][4];
    int nrej = 0;
    // After the first rejection at a node the register slice holds the unnormalised
    // residual r instead of the logits; the current p is r * pscale.
    bool lv_is_p = false;
    float pscale = 0.0f;
    float M = 0.0f, MC = 0.0f;  // raw max logit of the row, fl(M c2)
    float invZf = 1.0f;         // 1 / sum of 2^(l c2 - MC): the passes' normaliser
    ff Qsum = ff_make(0.0f);
    int amax = 0;

    while (!err) {
        if (!TSV_IN_BOUNDS(node, N, a.seq_err + b)) {
            err = TSV_DERR_INTERNAL;
            break;
        }
        const TL* lrow = static_cast<const TL*>(a.logits) + ((long long)b * N + node) * V;
        const float* qrow = greedy ? nullptr : a.probs + ((long long)b * N + node) * V;
        // children of `node`, in index order, and their scalars' buffers for this node
        const int nk = s_kcnt[node];
        const int* kids = s_kidlist + s_kstart[node];
        float* s_lx = s_lx2 + (plen & 1) * kMaxNodes;
        float* s_qx = s_qx2 + (plen & 1) * kMaxNodes;
        float* s_ux = s_ux2 + (plen & 1) * kMaxNodes;
        // the last warp starts asynchronous copies of the scalars the children's tests
        // need (they land while the row is reduced); the rest of the block starts on the row
        if (warp == nwarps - 1) {
            for (int t = lane; t < nk; t += 32) {
                const int x = s_tok[kids[t]];
                s_qx[t] = 0.0f;
                if (x >= 0 && x < V) {
                    if (sizeof(TL) == 4)
                        cp_async4(&s_lx[t], lrow + x);
                    else
                        s_lx[t] = to_f32(lrow[x]);  // 2-byte entries: a plain load
                    if (!greedy) {
                        cp_async4(&s_qx[t], qrow + x);
                        cp_async4(&s_ux[t], a.u_accept + (long long)b * N + kids[t]);
                    }
                }
            }
            cp_async_commit();
        }
        load_slice<VEC, ALIGNED>(lrow, v0, v1, lv, -INFINITY);
        // the first child's logits row into L2, for the likely case that it is accepted
        if (nk > 0) prefetch_slice<VEC>(static_cast<const TL*>(a.logits) + ((long long)b * N + kids[0]) * V, v0, v1);

        int bad = 0;
#pragma unroll
        for (int k = 0; k < VEC; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                if (v < v1 && !isfinite(lv[k][e])) bad = 1;
            }

        if (greedy) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                    if (v < v1 && (lv[k][e] > bv || (lv[k][e] == bv && v < bi))) {
                        bv = lv[k][e];
                        bi = v;
                    }
                }
            warp_argmax(bv, bi);
            bad = warp_or(bad);
            if (lane == 0) {
                s_wf[warp] = bv;
                s_wi[warp] = bi;
                s_wb[warp] = bad;
            }
            __syncthreads();
            if (warp == 0) {
                float v = lane < nwarps ? s_wf[lane] : -INFINITY;
                int i = lane < nwarps ? s_wi[lane] : 0x7fffffff;
                const int f = warp_or(lane < nwarps ? s_wb[lane] : 0);
                warp_argmax(v, i);
                if (lane == 0) {
                    RedSlot m{};
                    m.a = v;
                    m.i = i;
                    m.flag = f;
                    s_cta = m;
                }
            }
            cluster_allreduce(cluster, s_red, parity, s_cta, kRedArgmax, c2, &s_all, true);
            parity ^= 1;
            amax = s_all.i;
        } else {
            // per warp: raw max m_w and sum of 2^(l c2 - fl(m_w c2)), fp32, 4 accumulators
            float m = -INFINITY;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) m = fmaxf(m, lv[k][e]);
            m = warp_max(m);
            float sacc = 0.0f;
            if (m > -INFINITY) {
                const float mc = m * c2;
                float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int k = 0; k < VEC; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s4[e] += ex2(fmaf(lv[k][e], c2, -mc));  // padding: 2^-inf = 0
                sacc = (s4[0] + s4[1]) + (s4[2] + s4[3]);
            }
            sacc = warp_sum(sacc);
            bad = warp_or(bad);
            if (lane == 0) {
                s_wf[warp] = m;
                s_wg[warp] = sacc;
                s_wb[warp] = bad;
            }
            __syncthreads();
            if (warp == 0) {
                const float wm = lane < nwarps ? s_wf[lane] : -INFINITY;
                const float ws = lane < nwarps ? s_wg[lane] : 0.0f;
                const int f = warp_or(lane < nwarps ? s_wb[lane] : 0);
                const float cm = warp_max(wm);
                ff c = ws > 0.0f ? ff_mul_f(ff_make(ws), exp2f(wm * c2 - cm * c2)) : ff_make(0.0f);
                c = warp_sum_ff(c);
                if (lane == 0) {
                    RedSlot r{};
                    r.a = cm;
                    r.hi = c.hi;
                    r.lo = c.lo;
                    r.flag = f;
                    s_cta = r;
                }
            }
            // warp 0, before the reduction's closing barrier: the children's p(x), q(x) at
            // level 0, one lane per child (p(x) in float-float from a compensated exponent
            // argument; the normaliser is Zf without the rounding of M c2).  The last warp's
            // copies of the children's scalars have landed by the cluster barrier.
            auto children_p = [&](const RedSlot& o) {
                const float Mo = o.a, MCo = Mo * c2;
                const ff Z = ff_mul_f(ff{o.hi, o.lo}, exp2f(-fmaf(Mo, c2, -MCo)));
                const ff invZ = ff_recip(Z);
                for (int t = lane; t < nk; t += 32) {
                    const float qraw = s_qx[t];
                    ff px = ff_make(0.0f);
                    if (isfinite(qraw)) {
                        const ff arg = ff_mul(two_sum(s_lx[t], -Mo), invT_ff);
                        const float ex = expf(arg.hi);
                        px = ff_mul(quick_two_sum(ex, ex * arg.lo), invZ);
                    }
                    s_px[t] = px;
                    s_qc[t] = ff_make(qraw);
                    s_rflag[t] = 0;
                }
            };
            cluster_allreduce(cluster, s_red, parity, s_cta, kRedStats, c2, &s_all, true, children_p);
            parity ^= 1;
            M = s_all.a;
            MC = M * c2;
            invZf = 1.0f / ff_float(ff{s_all.hi, s_all.lo});
        }
        if (s_all.flag) {
            err = TSV_DERR_NONFINITE;
            break;
        }
        if (!greedy && filtered) {
            // ---- top-k / top-p filtered target (Sequoia summary, "More on tables"): keep the
            // first entries of the row in order of decreasing p (= decreasing logit; ties to
            // the lower index) up to the first position where their number reaches top_k or
            // their unfiltered mass reaches top_p; renormalise over them.  The boundary
            // entry's order key is found bit by bit (every probe one cluster reduction of a
            // count and a float-float mass, identical in every CTA), a partial run of equal
            // logits at the boundary is cut by index the same way.
            const ff pt = ff_make(a.top_p < 1.0f ? a.top_p : 3.0e38f);
            auto cond = [&](float cnt, ff mass) { return cnt >= kt || !ff_lt(mass, pt); };
            uint32_t theta = 0u;
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t cand = theta | (1u << bit);
                float cn = 0.0f, ms = 0.0f;
#pragma unroll
                for (int k = 0; k < VEC; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                        if (v < v1 && order_key(lv[k][e]) >= cand) {
                            cn += 1.0f;
                            ms += ex2(fmaf(lv[k][e], c2, -MC)) * invZf;
                        }
                    }
                reduce_sums(cn, ms);
                if (cond(s_all.hi, ff{s_all.hi2, s_all.lo2})) theta = cand;
            }
            // entries above the boundary key, and the run of entries equal to it
            float ca = 0.0f, ma = 0.0f, ct = 0.0f;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                    if (v >= v1) continue;
                    const uint32_t key = order_key(lv[k][e]);
                    if (key > theta) {
                        ca += 1.0f;
                        ma += ex2(fmaf(lv[k][e], c2, -MC)) * invZf;
                    } else if (key == theta) {
                        ct += 1.0f;
                    }
                }
            reduce_sums(ca, ma);
            const float c_above = s_all.hi;
            const ff m_above{s_all.hi2, s_all.lo2};
            reduce_sums(ct, 0.0f);
            const int n_tie = (int)s_all.hi;
            // how many of the tied entries the cut keeps (all CTAs compute the same)
            const float p_tie = ex2(fmaf(order_key_value(theta), c2, -MC)) * invZf;
            int keep_ties = n_tie;
            if (a.top_k > 0) keep_ties = min(keep_ties, max(1, (int)(kt - c_above)));
            if (a.top_p < 1.0f) {
                int tp = 1;
                while (tp < keep_ties && ff_lt(ff_add(m_above, ff_mul_f(ff_make((float)tp), p_tie)), pt)) ++tp;
                keep_ties = min(keep_ties, tp);
            }
            int idx_end = V;  // tied entries with index < idx_end are kept
            if (keep_ties < n_tie) {
                // index of the keep_ties-th tied entry: the largest bound with fewer ties below it
                int bound = 0;
                for (int bit = 20; bit >= 0; --bit) {
                    const int cand = bound | (1 << bit);
                    float cn = 0.0f;
#pragma unroll
                    for (int k = 0; k < VEC; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                            if (v < v1 && v < cand && order_key(lv[k][e]) == theta) cn += 1.0f;
                        }
                    reduce_sums(cn, 0.0f);
                    if ((int)s_all.hi < keep_ties) bound = cand;
                }
                idx_end = bound + 1;
            }
            // drop the rest and renormalise over the kept entries
            float zk = 0.0f;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                    const uint32_t key = order_key(lv[k][e]);
                    const bool kept = v < v1 && (key > theta || (key == theta && v < idx_end));
                    if (!kept) lv[k][e] = -INFINITY;
                    else zk += ex2(fmaf(lv[k][e], c2, -MC));
                }
            reduce_sums(zk, 0.0f);
            const ff zkeep{s_all.hi, s_all.lo};
            invZf = 1.0f / ff_float(zkeep);
            if (warp == 0) {  // the children's p(x) under the filtered target
                const ff invZ = ff_recip(ff_mul_f(zkeep, exp2f(-fmaf(M, c2, -MC))));
                for (int t = lane; t < nk; t += 32) {
                    const int x = s_tok[kids[t]];
                    const float lx = s_lx[t];
                    const uint32_t key = order_key(lx);
                    const bool kept = key > theta || (key == theta && x < idx_end);
                    ff px = ff_make(0.0f);
                    if (kept && isfinite(s_qx[t])) {
                        const ff arg = ff_mul(two_sum(lx, -M), invT_ff);
                        const float ex = expf(arg.hi);
                        px = ff_mul(quick_two_sum(ex, ex * arg.lo), invZ);
                    }
                    s_px[t] = px;
                }
            }
            __syncthreads();
        }

        // ---- children, in index order
        nrej = 0;
        lv_is_p = false;
        bool q_loaded = false;
        int next = -1;
        for (int t = 0; t < nk; ++t) {
            const int c = kids[t];
            const int x = s_tok[c];
            if (x < 0 || x >= V) {
                err = TSV_DERR_TOKEN;
                break;
            }
            if (greedy) {
                if (x == amax) {
                    next = c;
                    break;
                }
                continue;
            }
            if (!isfinite(s_qx[t])) {
                err = TSV_DERR_NONFINITE;
                break;
            }
            // u < p/q, i.e. u * q < p (q > 0); q == 0 accepts iff p > 0
            const ff px = s_px[t], qx = s_qc[t];
            const bool accept = ff_pos(qx) ? ff_lt(ff_mul_f(qx, s_ux[t]), px) : ff_pos(px);
            if (accept) {
                next = c;
                break;
            }
            // rejected: residual sum at the next level (and, the first time, sum q)
            int qb = 0;
            // q at this level: the raw row at the node's first pass, and throughout when
            // siblings were drafted independently (with replacement q is never updated)
            const bool raw_q = nrej == 0 || a.replacement;
            const uint64_t excl = raw_q ? 0ull : owned_mask<VEC>(s_xrej, nrej, v0, v1);  // tokens out of q here
            const float inv_sq = raw_q ? 1.0f : s_inv_sq[nrej];
            float zr = 0.0f, qs = 0.0f;
            constexpr int QG = VEC < 4 ? VEC : 4;  // draft entries loaded per group of vector steps
#pragma unroll
            for (int k0 = 0; k0 < VEC; k0 += QG) {
                float qk[QG][4];
#pragma unroll
                for (int kk = 0; kk < QG; ++kk) {
                    const int off = ((k0 + kk) * (int)blockDim.x + tid) * 4;
                    if (bulk && nrej > 0) {  // kept by this node's first pass
                        float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        if (v0 + off < v1) t = *reinterpret_cast<const float4*>(s_q + off);
                        qk[kk][0] = t.x;
                        qk[kk][1] = t.y;
                        qk[kk][2] = t.z;
                        qk[kk][3] = t.w;
                    } else {
                        load4<ALIGNED>(qrow, v0 + off, v1, qk[kk], 0.0f);
                        if (bulk && v0 + off < v1)
                            *reinterpret_cast<float4*>(s_q + off) = make_float4(qk[kk][0], qk[kk][1], qk[kk][2], qk[kk][3]);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < QG; ++kk) {
                    const int k = k0 + kk;
                    const int base = v0 + (k * (int)blockDim.x + tid) * 4;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int v = base + e;
                        const float q = qk[kk][e];
                        if (v < v1 && !isfinite(q)) qb = 1;
                        // p and q at the current level
                        const float p = lv_is_p ? lv[k][e] * pscale : ex2(fmaf(lv[k][e], c2, -MC)) * invZf;
                        const float qc = raw_q ? q : (((excl >> (k * 4 + e)) & 1ull) ? 0.0f : q * inv_sq);
                        const float d = fmaxf(0.0f, p - qc);
                        zr += d;
                        qs += q;
                        lv[k][e] = (v < v1) ? d : 0.0f;  // the residual replaces the slice
                    }
                }
            }
            zr = warp_sum(zr);
            qs = warp_sum(qs);
            qb = warp_or(qb);
            if (lane == 0) {
                s_wf[warp] = zr;
                s_wg[warp] = qs;
                s_wb[warp] = qb;
            }
            __syncthreads();
            if (warp == 0) {
                const ff z1 = warp_sum_ff(ff_make(lane < nwarps ? s_wf[lane] : 0.0f));
                const ff z2 = warp_sum_ff(ff_make(lane < nwarps ? s_wg[lane] : 0.0f));
                const int f = warp_or(lane < nwarps ? s_wb[lane] : 0);
                if (lane == 0) {
                    RedSlot r{};
                    r.hi = z1.hi;
                    r.lo = z1.lo;
                    r.hi2 = z2.hi;
                    r.lo2 = z2.lo;
                    r.flag = f;
                    s_cta = r;
                }
            }
            cluster_allreduce(cluster, s_red, parity, s_cta, kRedSums, c2, &s_all);
            parity ^= 1;
            if (s_all.flag) {
                err = TSV_DERR_NONFINITE;
                break;
            }
            if (!q_loaded) Qsum = ff{s_all.hi2, s_all.lo2};
            q_loaded = true;
            // level j = nrej + 1: its residual sum Zr_j and S_j = sum of q without the
            // distinct rejected tokens; then every later child's (p, q) moves to level j
            const int j = nrej + 1;
            const ff zr_new{s_all.hi, s_all.lo};
            if (warp == 0) {
                bool dup = false;
                for (int i2 = lane; i2 < nrej; i2 += 32) dup |= (s_xrej[i2] == x);
                dup = __any_sync(0xffffffffu, dup);
                const ff sq = dup ? (j == 1 ? Qsum : s_sq[j - 1]) : ff_sub(j == 1 ? Qsum : s_sq[j - 1], ff_make(s_qx[t]));
                const bool zr_ok = ff_pos(zr_new);
                __syncwarp();
                if (lane == 0) {
                    s_xrej[j - 1] = x;
                    s_zr[j] = zr_new;
                    s_zr_ok[j] = zr_ok;
                    s_inv_zr[j] = zr_ok ? ff_float(ff_div(ff_make(1.0f), zr_new)) : 1.0f;
                    s_sq[j] = sq;
                    s_inv_sq[j] = ff_pos(sq) ? ff_float(ff_div(ff_make(1.0f), sq)) : 0.0f;
                }
                const ff inv_zr = zr_ok ? ff_recip(zr_new) : ff_make(1.0f);
                const ff inv_sq = ff_pos(sq) ? ff_recip(sq) : ff_make(0.0f);
                for (int t2 = t + 1 + lane; t2 < nk; t2 += 32) {
                    ff p2 = s_px[t2];
                    const ff q2 = s_qc[t2];
                    if (zr_ok) p2 = ff_mul(ff_max0(ff_sub(p2, q2)), inv_zr);
                    int rf = s_rflag[t2];
                    if (s_tok[kids[t2]] == x) rf = 1;
                    s_px[t2] = p2;
                    if (!a.replacement)  // with replacement the later children keep the raw q(x)
                        s_qc[t2] = (rf || !ff_pos(sq)) ? ff_make(0.0f) : ff_mul_f(inv_sq, s_qx[t2]);
                    s_rflag[t2] = rf;
                }
            }
            __syncthreads();
            ++nrej;
            if (s_zr_ok[nrej]) {
                lv_is_p = true;
                pscale = s_inv_zr[nrej];
            } else {
                // empty residual: p keeps its previous value, which the pass overwrote --
                // rebuild it from the logits (unreachable in exact arithmetic)
                rebuild_level<VEC, ALIGNED>(lv, lrow, qrow, v0, v1, nrej, c2, MC, invZf, s_xrej, s_inv_sq, s_inv_zr,
                                            s_zr_ok, a.replacement != 0);
                lv_is_p = true;
                pscale = 1.0f;
            }
        }
        if (err || next < 0) break;
        // no block barrier here: the next node's copies go to the other buffers, and everything
        // else it writes before its first barrier is read by this node only before one
        if (tid == 0) s_path[plen] = next;
        ++plen;
        node = next;
    }

    if (warp == nwarps - 1) asm volatile("cp.async.wait_all;" ::: "memory");  // no copies in flight at exit

    // ---- outputs
    const long long rowoff = (long long)b * N;
    if (err) {
        if (rank == 0) {
            for (int j = tid; j < N; j += blockDim.x) {
                a.accepted_nodes[rowoff + j] = -1;
                a.out_tokens[rowoff + j] = -1;
            }
            if (tid == 0) {
                a.accept_len[b] = -1;
                a.bonus_token[b] = -1;
                a.seq_err[b] = err;
            }
        }
        cluster.sync();
        if (a.k_cache && rank == 0) fused_compact(a, b, -1, s_path, &s_flag, s_path, s_blkerr);
        return;
    }
    if (rank == 0) {
        for (int j = tid; j < N; j += blockDim.x) {
            a.accepted_nodes[rowoff + j] = j < plen ? s_path[j] : -1;
            a.out_tokens[rowoff + j] =
                (j + 1 < plen && TSV_IN_BOUNDS(s_path[j + 1], N, a.seq_err + b)) ? s_tok[s_path[j + 1]] : -1;
        }
        if (tid == 0) {
            a.accept_len[b] = plen - 1;
            a.seq_err[b] = 0;
        }
    }
    if (greedy) {
        if (rank == 0 && tid == 0) {
            a.bonus_token[b] = amax;
            a.out_tokens[rowoff + plen - 1] = amax;
        }
        cluster.sync();
        if (a.k_cache && rank == 0) fused_compact(a, b, plen - 1, s_path, &s_flag, s_path, s_blkerr);
        return;
    }

    // ---- bonus: inverse CDF of the current p in token order.  Token order within a
    // CTA is (vector step k, warp, lane, element); prefix sums are float-float.
    float(&pk)[VEC][4] = lv;  // the slice is not needed after this pass
#pragma unroll
    for (int k = 0; k < VEC; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
            const float p = lv_is_p ? lv[k][e] * pscale : ex2(fmaf(lv[k][e], c2, -MC)) * invZf;
            pk[k][e] = (v < v1) ? p : 0.0f;
        }
    if (!(a.u_bonus[b] < 1.0f)) {
        // u at or past the top of [0, 1) (or NaN): no CDF boundary lies above it, so the
        // draw is the inverse CDF's limit there, the last token with p > 0 (the same
        // rule as the oracle's)
        int last = -1;
#pragma unroll
        for (int k = 0; k < VEC; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                if (v < v1 && pk[k][e] > 0.0f) last = max(last, v);
            }
        float lv_ = last >= 0 ? (float)last : -INFINITY;  // indices < 2^24 are exact in fp32
        warp_argmax(lv_, last);
        if (lane == 0) {
            s_wf[warp] = lv_;
            s_wi[warp] = last;
        }
        __syncthreads();
        if (warp == 0) {
            float v = lane < nwarps ? s_wf[lane] : -INFINITY;
            int i = lane < nwarps ? s_wi[lane] : -1;
            warp_argmax(v, i);
            if (lane == 0) {
                RedSlot m{};
                m.a = v;
                m.i = i;
                s_cta = m;
            }
        }
        cluster_allreduce(cluster, s_red, parity, s_cta, kRedArgmax, c2, &s_all);
        parity ^= 1;
        if (rank == 0 && tid == 0) {
            const int tok = s_all.a > -INFINITY ? s_all.i : -1;
            a.bonus_token[b] = tok;
            a.out_tokens[rowoff + plen - 1] = tok;
        }
        cluster.sync();
        if (a.k_cache && rank == 0) fused_compact(a, b, plen - 1, s_path, &s_flag, s_path, s_blkerr);
        return;
    }
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const float ts = warp_sum(pk[k][0] + pk[k][1] + pk[k][2] + pk[k][3]);
        if (lane == 0) s_seg[k * nwarps + warp] = ts;
    }
    __syncthreads();
    const int nseg = VEC * nwarps;
    if (warp == 0) {
        // each lane owns a run of consecutive segments.  Each level's exclusive base is
        // the previous level's inclusive value itself (never a difference), so the
        // intervals tile [0, total) exactly.
        const int per = (nseg + 31) / 32;
        ff run = ff_make(0.0f);
        for (int s2 = lane * per; s2 < min(nseg, lane * per + per); ++s2) run = ff_add(run, ff_make(s_seg[s2]));
        ff incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const ff y{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
            if (lane >= o) incl = ff_add(incl, y);
        }
        ff base{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
        if (lane == 0) base = ff_make(0.0f);
        for (int s2 = lane * per; s2 < min(nseg, lane * per + per); ++s2) {
            base = ff_add(base, ff_make(s_seg[s2]));
            s_segcum[s2] = base;
        }
    }
    __syncthreads();
    if (tid == 0) {
        RedSlot r{};
        r.hi = s_segcum[nseg - 1].hi;  // CTA total
        r.lo = s_segcum[nseg - 1].lo;
        s_red[parity * kMaxCluster] = r;
    }
    cluster.sync();
    if (warp == 0) {
        ff tot = ff_make(0.0f);
        if (lane < cs) {
            const RedSlot* rs = cluster.map_shared_rank(&s_red[parity * kMaxCluster], lane);
            tot = ff{rs->hi, rs->lo};
        }
        ff incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const ff y{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
            if (lane >= o) incl = ff_add(incl, y);
        }
        ff excl{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
        if (lane == 0) excl = ff_make(0.0f);
        const ff grand{__shfl_sync(0xffffffffu, incl.hi, cs - 1), __shfl_sync(0xffffffffu, incl.lo, cs - 1)};
        const ff mine_incl{__shfl_sync(0xffffffffu, incl.hi, rank), __shfl_sync(0xffffffffu, incl.lo, rank)};
        const ff mine_excl{__shfl_sync(0xffffffffu, excl.hi, rank), __shfl_sync(0xffffffffu, excl.lo, rank)};
        if (lane == 0) {
            const ff target = ff_mul_f(grand, a.u_bonus[b]);  // u in [0,1): target < grand
            s_target = ff_sub(target, mine_excl);
            s_claim = (!ff_lt(target, mine_excl) && ff_lt(target, mine_incl)) ? 1 : 0;
        }
    }
    parity ^= 1;
    __syncthreads();
    if (s_claim) {
        // this CTA holds the crossing: find the segment, then the lane, then the element
        if (tid == 0) {
            const ff target = s_target;
            int seg = -1;
            for (int s2 = 0; s2 < nseg; ++s2)
                if (ff_lt(target, s_segcum[s2])) {
                    seg = s2;
                    break;
                }
            if (seg < 0)  // only by rounding of the base subtraction: last segment with mass
                for (int s2 = nseg - 1; s2 >= 0 && seg < 0; --s2)
                    if (s_seg[s2] > 0.0f) seg = s2;
            s_segsel = seg;
            s_target = seg > 0 ? ff_sub(target, s_segcum[seg - 1]) : target;
        }
        __syncthreads();
        const int seg = s_segsel;
        const int kseg = seg / nwarps, wseg = seg % nwarps;
        if (warp == wseg) {
            const float tgt = ff_float(s_target);
            float pe[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if (k == kseg) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) pe[e] = pk[k][e];
                }
            const float ts = pe[0] + pe[1] + pe[2] + pe[3];
            float incl = ts;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.0f;
            const unsigned hit = __ballot_sync(0xffffffffu, tgt < incl && ts > 0.0f);
            const unsigned has = __ballot_sync(0xffffffffu, ts > 0.0f);
            // fp32 rounding can leave no lane past the target: take the last with mass
            const int l_sel = hit ? (__ffs(hit) - 1) : (31 - __clz(has));
            if (lane == l_sel) {
                float cum = excl;
                int e_sel = -1, e_last = -1;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (pe[e] > 0.0f) e_last = e;
                    cum += pe[e];
                    if (e_sel < 0 && tgt < cum && pe[e] > 0.0f) e_sel = e;
                }
                if (e_sel < 0) e_sel = e_last;
                const int tok = v0 + (kseg * (int)blockDim.x + tid) * 4 + e_sel;
                (void)TSV_IN_BOUNDS(tok, V, a.seq_err + b);  // a drawn token outside the vocabulary
                a.bonus_token[b] = tok;
                a.out_tokens[rowoff + plen - 1] = tok;
            }
        }
    }
    cluster.sync();
    if (a.k_cache && rank == 0) fused_compact(a, b, plen - 1, s_path, &s_flag, s_path, s_blkerr);
}

}  // namespace tsv

namespace tsv {

// dynamic shared memory of the walk: aligned rows keep the node's draft row slice
// (v_per_cta floats)
template <bool ALIGNED>
static size_t reject_smem(int vpc) {
    return ALIGNED ? (size_t)vpc * sizeof(float) : 0;
}

template <int VEC, bool ALIGNED, typename TL>
static cudaError_t make_reject_config(int B, int cs, int threads, int vpc, cudaStream_t stream,
                                      cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr) {
    cudaError_t e = cudaFuncSetAttribute(tree_reject_kernel<VEC, ALIGNED, TL>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    const size_t smem = reject_smem<ALIGNED>(vpc);
    e = cudaFuncSetAttribute(tree_reject_kernel<VEC, ALIGNED, TL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3((unsigned)(B * cs), 1, 1);
    cfg->blockDim = dim3((unsigned)threads, 1, 1);
    cfg->dynamicSmemBytes = smem;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
    return cudaSuccess;
}

template <int VEC, bool ALIGNED, typename TL>
static cudaError_t launch_reject_inst(const SampleArgs& a, int B, int cs, int threads, cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    cudaError_t e = make_reject_config<VEC, ALIGNED, TL>(B, cs, threads, a.v_per_cta, stream, &cfg, attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(tree_reject_kernel<VEC, ALIGNED, TL>, cfg.gridDim, cfg.blockDim, cfg.dynamicSmemBytes, stream,
                      static_cast<unsigned>(cs), a);
}

// How many clusters of this shape can be resident at once (cached per shape).
template <int VEC, bool ALIGNED, typename TL>
static int resident_clusters(int cs, int threads, int vpc) {
    static std::mutex mu;
    static std::map<std::pair<long long, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(((long long)dev * 64 + cs) * (1LL << 32) + vpc, threads);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    int n = 0;
    if (make_reject_config<VEC, ALIGNED, TL>(1, cs, threads, vpc, nullptr, &cfg, attr) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, tree_reject_kernel<VEC, ALIGNED, TL>, &cfg) != cudaSuccess)
        n = 0;
    cache[key] = n;
    return n;
}

static int vec_for(int V, int cs, int threads, int* vpc_out, bool allow16 = false) {
    int vpc = (V + cs - 1) / cs;
    vpc = (vpc + 3) & ~3;
    *vpc_out = vpc;
    const int need = (vpc + threads * 4 - 1) / (threads * 4);
    return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 8 ? 8 : (allow16 && need <= 16) ? 16 : 0;
}

template <bool ALIGNED, typename TL>
static int resident_for(int vec, int cs, int threads, int vpc) {
    switch (vec) {
        case 1: return resident_clusters<1, ALIGNED, TL>(cs, threads, vpc);
        case 2: return resident_clusters<2, ALIGNED, TL>(cs, threads, vpc);
        case 4: return resident_clusters<4, ALIGNED, TL>(cs, threads, vpc);
        case 16: return resident_clusters<16, ALIGNED, TL>(cs, threads, vpc);
        default: return resident_clusters<8, ALIGNED, TL>(cs, threads, vpc);
    }
}

template <bool ALIGNED, typename TL>
static cudaError_t launch_vec(const SampleArgs& a, int vec, int B, int cs, int threads, cudaStream_t stream) {
    switch (vec) {
        case 1: return launch_reject_inst<1, ALIGNED, TL>(a, B, cs, threads, stream);
        case 2: return launch_reject_inst<2, ALIGNED, TL>(a, B, cs, threads, stream);
        case 4: return launch_reject_inst<4, ALIGNED, TL>(a, B, cs, threads, stream);
        case 8: return launch_reject_inst<8, ALIGNED, TL>(a, B, cs, threads, stream);
        case 16: return launch_reject_inst<16, ALIGNED, TL>(a, B, cs, threads, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Chooses the cluster size, block size and per-thread vector count for a vocabulary of
// V entries and B sequences, then launches one cluster per sequence (16-CTA clusters
// need 16 free SMs in one GPC, so their residency is checked).
template <typename TL>
static cudaError_t launch_tree_reject_t(SampleArgs a, int B, int num_sms, cudaStream_t stream) {
    const int V = a.V;
    int threads = 64;
    while (threads < 512 && threads * 4 * 2 < V) threads *= 2;
    const int cap1 = threads * 4 * 8;  // entries one CTA holds at VEC = 8
    int cs_min = 1;
    while (cs_min * cap1 < V) cs_min *= 2;  // smallest cluster that fits the row
    // aligned: four entries per vector load start on a 16-byte (fp32) / 8-byte (bf16) boundary
    const bool aligned = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & (4 * sizeof(TL) - 1)) == 0 &&
                         (a.probs == nullptr || (reinterpret_cast<uintptr_t>(a.probs) & 15) == 0);
    // Enough CTAs that a thread holds at most 8 entries: every visited node costs a
    // pass over the slice, and the slice load dominates it.  A cluster larger than the
    // smallest that fits the row is kept only if all B clusters can be resident at once
    // (sizes between powers of two are tried too: 16-CTA clusters need 16 free SMs in
    // one GPC, which not every GPC has).
    int cs = cs_min;
    while (cs < 16 && cs * threads * 8 < V) cs *= 2;
    for (; cs > cs_min; --cs) {
        int vpc;
        const int vec = vec_for(V, cs, threads, &vpc);
        if (vec == 0) continue;
        const int res =
            aligned ? resident_for<true, TL>(vec, cs, threads, vpc) : resident_for<false, TL>(vec, cs, threads, vpc);
        if (res >= B && B * cs <= num_sms) break;
    }
    int vpc;
    int vec = vec_for(V, cs, threads, &vpc);
    // When the B clusters do not fit at once, 384-thread CTAs with 16 vector steps a thread
    // (168 registers) hold 1.5x the entries per SM, so more sequences walk at the same time;
    // a node then costs a little more (a larger slice per CTA), but most of its cost is
    // latency, so this pays once the resident clusters grow by a fifth.
    if (threads == 512 && vec == 8) {
        const int res8 =
            aligned ? resident_for<true, TL>(vec, cs, threads, vpc) : resident_for<false, TL>(vec, cs, threads, vpc);
        int cs16 = 1;
        while (cs16 < 16 && cs16 * 384 * 4 * 16 < V) ++cs16;
        int vpc16;
        const int vec16 = vec_for(V, cs16, 384, &vpc16, true);
        if (res8 < B && vec16 == 16) {
            const int res16 = aligned ? resident_for<true, TL>(vec16, cs16, 384, vpc16)
                                      : resident_for<false, TL>(vec16, cs16, 384, vpc16);
            if (5 * res16 >= 6 * res8) {
                threads = 384;
                cs = cs16;
                vec = vec16;
                vpc = vpc16;
            }
        }
    }
    a.v_per_cta = vpc;
    return aligned ? launch_vec<true, TL>(a, vec, B, cs, threads, stream)
                   : launch_vec<false, TL>(a, vec, B, cs, threads, stream);
}

cudaError_t launch_tree_reject(SampleArgs a, int B, int num_sms, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    return a.logits_bf16 ? launch_tree_reject_t<__nv_bfloat16>(a, B, num_sms, stream)
                         : launch_tree_reject_t<float>(a, B, num_sms, stream);
}

}  // namespace tsv
