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
// (fp32) -> one warp per CTA (fp64) -> DSMEM across the cluster (fp64); every CTA
// combines the cluster partials in the same order, so all CTAs hold bit-identical
// scalars and take identical decisions without a second exchange.  The rows of the
// current node's children and its draft row are prefetched into L2 while the
// current row is reduced.  The p(x)/q(x) ratio is evaluated in fp64 from the
// reduced scalars.
#include <cooperative_groups.h>

#include "common.cuh"
#include "verify_args.cuh"

namespace cg = cooperative_groups;

namespace tsv {

struct __align__(16) RedSlot {
    double a;
    double b;
    int i;
    int flag;
};

constexpr int kMaxRejections = kMaxNodes;  // at most one per tried child

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
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_max_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
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
        float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (v2 > v || (v2 == v && i2 < i)) {
            v = v2;
            i = i2;
        }
    }
}

// true iff v is one of the first j rejected tokens xr[0..j-1]
__device__ __forceinline__ bool is_rejected(int v, int j, const int* xr) {
    for (int i = 0; i < j; ++i)
        if (xr[i] == v) return true;
    return false;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <int VEC, bool ALIGNED>
__device__ __forceinline__ void load_slice(const float* row, int v0, int v1, float (&x)[VEC][4], float fill) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int base = v0 + (k * (int)blockDim.x + (int)threadIdx.x) * 4;
        if (ALIGNED) {
            if (base < v1) {
                float4 t = __ldg(reinterpret_cast<const float4*>(row + base));
                x[k][0] = t.x;
                x[k][1] = t.y;
                x[k][2] = t.z;
                x[k][3] = t.w;
            } else {
                x[k][0] = x[k][1] = x[k][2] = x[k][3] = fill;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[k][e] = (base + e < v1) ? __ldg(row + base + e) : fill;
        }
    }
}

template <int VEC>
__device__ __forceinline__ void prefetch_slice(const float* row, int v0, int v1) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int base = v0 + (k * (int)blockDim.x + (int)threadIdx.x) * 4;
        // one prefetch per 128-byte line: every 8th thread of a coalesced float4 run
        if (base < v1 && ((reinterpret_cast<uintptr_t>(row + base) & 127) < 16)) prefetch_l2(row + base);
    }
}

template <int VEC, bool ALIGNED>
__global__ void __launch_bounds__(512, 1) tree_reject_kernel(const SampleArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int N = a.N, V = a.V;
    const int v0 = min(V, rank * a.v_per_cta), v1 = min(V, v0 + a.v_per_cta);
    const bool greedy = (a.T == 0.0f);
    const double Td = (double)a.T;

    __shared__ int s_par[kMaxNodes], s_tok[kMaxNodes], s_path[kMaxNodes];
    __shared__ int s_kids[kMaxNodes];
    __shared__ float s_lx[kMaxNodes], s_qx[kMaxNodes], s_ux[kMaxNodes];
    __shared__ RedSlot s_red[2];
    __shared__ float s_wf[32], s_wg[32];
    __shared__ int s_wi[32], s_wb[32];
    __shared__ double s_res[4];
    __shared__ int s_ires[4];
    __shared__ int s_flag;
    // rejection history at the current node
    __shared__ int s_xrej[kMaxRejections];        // rejected tokens x_1.. at the current node
    __shared__ float s_qrej[kMaxRejections];      // their raw draft probabilities
    __shared__ double s_zr[kMaxRejections + 1];   // residual sums Zr_j (level j >= 1)
    __shared__ double s_sq[kMaxRejections + 1];   // S_j = sum of q over tokens not in {x_1..x_j}
    __shared__ float s_inv_zr[kMaxRejections + 1], s_inv_sq[kMaxRejections + 1];
    __shared__ int s_zr_ok[kMaxRejections + 1];

    int parity = 0;
    // Cluster all-reduce of one (a, b, i, flag) partial per CTA.  kind 0: (max, rescaled
    // sum) softmax statistics; kind 1: (sum, sum); kind 2: argmax (value in a, index in i).
    // Called by all threads of all CTAs.  Result in s_res[0..1], s_ires[0], s_ires[1].
    auto cluster_combine = [&](double pa, double pb, int pi, int pflag, int kind) {
        if (tid == 0) s_red[parity] = RedSlot{pa, pb, pi, pflag};
        cluster.sync();
        if (warp == 0) {
            double ra = (kind == 1) ? 0.0 : -INFINITY, rb = 0.0;
            int ri = 0x7fffffff, rf = 0;
            if (lane < cs) {
                const RedSlot* rs = cluster.map_shared_rank(&s_red[parity], lane);
                ra = rs->a;
                rb = rs->b;
                ri = rs->i;
                rf = rs->flag;
            }
            rf = warp_or(rf);
            if (kind == 0) {
                double m = warp_max_d(ra);
                double s = (lane < cs && rb > 0.0) ? rb * exp((ra - m) / Td) : 0.0;
                s = warp_sum_d(s);
                ra = m;
                rb = s;
            } else if (kind == 1) {
                ra = warp_sum_d(ra);
                rb = warp_sum_d(rb);
            } else {
                float fv = (float)ra;
                warp_argmax(fv, ri);
                ra = fv;
            }
            if (lane == 0) {
                s_res[0] = ra;
                s_res[1] = rb;
                s_ires[0] = ri;
                s_ires[1] = rf;
            }
        }
        parity ^= 1;
        __syncthreads();
    };

    // ---- tree and tokens
    for (int i = tid; i < N; i += blockDim.x) {
        s_par[i] = a.parent[(long long)b * N + i];
        s_tok[i] = a.tokens[(long long)b * N + i];
    }
    bool tree_ok = block_tree_ok(a.parent + (long long)b * N, N, &s_flag);

    int err = tree_ok ? 0 : TSV_DERR_PARENT;
    int node = 0, plen = 1;
    if (tid == 0) s_path[0] = 0;
    float lv[VEC][4], qv[VEC][4];
    int nrej = 0;
    bool q_loaded = false;
    double M = 0.0, Z = 1.0, Qsum = 0.0;
    int amax = 0;

    while (!err) {
        const float* lrow = a.logits + ((long long)b * N + node) * V;
        const float* qrow = greedy ? nullptr : a.probs + ((long long)b * N + node) * V;
        // children of `node`, in index order (identical in every thread)
        if (tid == 0) {
            int nk = 0;
            for (int c = node + 1; c < N; ++c)
                if (s_par[c] == node) s_kids[nk++] = c;
            s_ires[2] = nk;
        }
        __syncthreads();
        const int nk = s_ires[2];
        // scalar fetches for the children's tests, issued before the row pass
        for (int t = tid; t < nk; t += blockDim.x) {
            const int x = s_tok[s_kids[t]];
            if (x >= 0 && x < V) {
                s_lx[t] = __ldg(lrow + x);
                if (!greedy) {
                    s_qx[t] = __ldg(qrow + x);
                    s_ux[t] = __ldg(a.u_accept + (long long)b * N + s_kids[t]);
                }
            }
        }
        load_slice<VEC, ALIGNED>(lrow, v0, v1, lv, -INFINITY);
        // prefetch the children's logits rows and this node's draft row into L2
        for (int t = 0; t < nk && t < 4; ++t)
            prefetch_slice<VEC>(a.logits + ((long long)b * N + s_kids[t]) * V, v0, v1);
        if (!greedy && nk > 0) prefetch_slice<VEC>(qrow, v0, v1);

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
                int f = lane < nwarps ? s_wb[lane] : 0;
                warp_argmax(v, i);
                f = warp_or(f);
                if (lane == 0) {
                    s_res[2] = v;
                    s_ires[3] = i;
                    s_flag = f;
                }
            }
            __syncthreads();
            cluster_combine(s_res[2], 0.0, s_ires[3], s_flag, 2);
            amax = s_ires[0];
        } else {
            float m = -INFINITY;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) m = fmaxf(m, lv[k][e]);
            m = warp_max(m);
            float s = 0.0f;
            if (m > -INFINITY) {
#pragma unroll
                for (int k = 0; k < VEC; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s += expf((lv[k][e] - m) / a.T);
            }
            s = warp_sum(s);
            bad = warp_or(bad);
            if (lane == 0) {
                s_wf[warp] = m;
                s_wg[warp] = s;
                s_wi[warp] = bad;
            }
            __syncthreads();
            if (warp == 0) {
                double wm = lane < nwarps ? (double)s_wf[lane] : -INFINITY;
                double ws = lane < nwarps ? (double)s_wg[lane] : 0.0;
                int f = lane < nwarps ? s_wi[lane] : 0;
                double cm = warp_max_d(wm);
                double cs_ = (ws > 0.0) ? ws * exp((wm - cm) / Td) : 0.0;
                cs_ = warp_sum_d(cs_);
                f = warp_or(f);
                if (lane == 0) {
                    s_res[2] = cm;
                    s_res[3] = cs_;
                    s_flag = f;
                }
            }
            __syncthreads();
            cluster_combine(s_res[2], s_res[3], 0, s_flag, 0);
            M = s_res[0];
            Z = s_res[1];
        }
        if (s_ires[1]) {
            err = TSV_DERR_NONFINITE;
            break;
        }

        // ---- children, in index order
        nrej = 0;
        q_loaded = false;
        int next = -1;
        const float invZ = (float)(1.0 / Z);
        const float Mf = (float)M;  // M is the max of float logits: exact
        for (int t = 0; t < nk; ++t) {
            const int c = s_kids[t];
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
            // q(x) at the current level and the fp64 ratio (thread 0; broadcast)
            if (tid == 0) {
                const float qraw = s_qx[t];
                int e2 = 0;
                double ratio = 0.0;
                if (!isfinite(qraw)) {
                    e2 = TSV_DERR_NONFINITE;
                } else {
                    double px = exp(((double)s_lx[t] - M) / Td) / Z;
                    double qx = (double)qraw;  // level 0: the raw draft probability
                    bool x_rejected = false;
                    for (int j = 1; j <= nrej; ++j) {
                        // level j-1 -> j: residual on p, x_j removed from q
                        if (s_zr_ok[j]) px = fmax(0.0, px - qx) / s_zr[j];
                        if (s_xrej[j - 1] == x) x_rejected = true;
                        qx = (x_rejected || !(s_sq[j] > 0.0)) ? 0.0 : (double)qraw / s_sq[j];
                    }
                    if (qx > 0.0)
                        ratio = px / qx;
                    else
                        ratio = (px > 0.0) ? INFINITY : 0.0;
                }
                s_ires[2] = e2;
                s_ires[3] = (e2 == 0 && (double)s_ux[t] < ratio) ? 1 : 0;
            }
            __syncthreads();
            const int e2 = s_ires[2], accept = s_ires[3];
            __syncthreads();
            if (e2) {
                err = e2;
                break;
            }
            if (accept) {
                next = c;
                break;
            }
            // rejected: residual sum at the next level (and, the first time, sum q)
            if (!q_loaded) {
                load_slice<VEC, ALIGNED>(qrow, v0, v1, qv, 0.0f);
                int qb = 0;
#pragma unroll
                for (int k = 0; k < VEC; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                        if (v < v1 && !isfinite(qv[k][e])) qb = 1;
                    }
                qb = warp_or(qb);
                if (lane == 0) s_wi[warp] = qb;
            } else if (lane == 0) {
                s_wi[warp] = 0;
            }
            float zr = 0.0f, qs = 0.0f;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
                    float p = expf((lv[k][e] - Mf) / a.T) * invZ;
                    float q = qv[k][e];
                    for (int j = 1; j <= nrej; ++j) {
                        const float qprev =
                            (j == 1) ? q : (is_rejected(v, j - 1, s_xrej) ? 0.0f : q * s_inv_sq[j - 1]);
                        if (s_zr_ok[j]) p = fmaxf(0.0f, p - qprev) * s_inv_zr[j];
                    }
                    const float qcur =
                        (nrej == 0) ? q : (is_rejected(v, nrej, s_xrej) ? 0.0f : q * s_inv_sq[nrej]);
                    zr += fmaxf(0.0f, p - qcur);
                    if (!q_loaded) qs += q;
                }
            zr = warp_sum(zr);
            qs = warp_sum(qs);
            if (lane == 0) {
                s_wf[warp] = zr;
                s_wg[warp] = qs;
            }
            __syncthreads();
            if (warp == 0) {
                double z1 = lane < nwarps ? (double)s_wf[lane] : 0.0;
                double z2 = lane < nwarps ? (double)s_wg[lane] : 0.0;
                int f = lane < nwarps ? s_wi[lane] : 0;
                z1 = warp_sum_d(z1);
                z2 = warp_sum_d(z2);
                f = warp_or(f);
                if (lane == 0) {
                    s_res[2] = z1;
                    s_res[3] = z2;
                    s_flag = f;
                }
            }
            __syncthreads();
            cluster_combine(s_res[2], s_res[3], 0, s_flag, 1);
            if (s_ires[1]) {
                err = TSV_DERR_NONFINITE;
                break;
            }
            if (!q_loaded) Qsum = s_res[1];
            q_loaded = true;
            // record level nrej+1 (every thread holds the same values)
            const double zr_new = s_res[0];
            __syncthreads();
            if (tid == 0) {
                const int j = nrej + 1;
                s_xrej[j - 1] = x;
                s_qrej[j - 1] = s_qx[t];
                s_zr[j] = zr_new;
                s_zr_ok[j] = zr_new > 0.0;
                s_inv_zr[j] = zr_new > 0.0 ? (float)(1.0 / zr_new) : 1.0f;
                double sq = Qsum;
                for (int i2 = 0; i2 < j; ++i2) {  // subtract each distinct rejected token once
                    bool dup = false;
                    for (int i3 = 0; i3 < i2; ++i3) dup |= (s_xrej[i3] == s_xrej[i2]);
                    if (!dup) sq -= (double)s_qrej[i2];
                }
                s_sq[j] = sq;
                s_inv_sq[j] = sq > 0.0 ? (float)(1.0 / sq) : 0.0f;
            }
            __syncthreads();
            ++nrej;
        }
        if (err || next < 0) break;
        if (tid == 0) s_path[plen] = next;
        ++plen;
        node = next;
        __syncthreads();
    }

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
        return;
    }
    if (rank == 0) {
        for (int j = tid; j < N; j += blockDim.x) {
            a.accepted_nodes[rowoff + j] = j < plen ? s_path[j] : -1;
            a.out_tokens[rowoff + j] = (j + 1 < plen) ? s_tok[s_path[j + 1]] : -1;
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
        return;
    }

    // ---- bonus: inverse CDF of the current p over token order
    // per-thread 4-element sums for every vector step k; token order within a CTA is
    // (k, warp, lane, element)
    const float invZ = (float)(1.0 / Z);
    float (&pk)[VEC][4] = lv;  // the logits slice is not needed after this pass
#pragma unroll
    for (int k = 0; k < VEC; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = v0 + (k * (int)blockDim.x + tid) * 4 + e;
            float p = expf((lv[k][e] - (float)M) / a.T) * invZ;
            const float q = qv[k][e];
            for (int j = 1; j <= nrej; ++j) {
                const float qprev = (j == 1) ? q : (is_rejected(v, j - 1, s_xrej) ? 0.0f : q * s_inv_sq[j - 1]);
                if (s_zr_ok[j]) p = fmaxf(0.0f, p - qprev) * s_inv_zr[j];
            }
            pk[k][e] = (v < v1) ? p : 0.0f;
        }
    __shared__ float s_seg[8 * 16];     // [k][warp] segment sums
    __shared__ double s_segcum[8 * 16];  // inclusive prefix over (k, warp)
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        float ts = pk[k][0] + pk[k][1] + pk[k][2] + pk[k][3];
        ts = warp_sum(ts);
        if (lane == 0) s_seg[k * nwarps + warp] = ts;
    }
    __syncthreads();
    const int nseg = VEC * nwarps;
    if (warp == 0) {
        // each lane owns a run of consecutive segments; fp64 prefix.  Each level's
        // exclusive base is the previous level's inclusive value itself (never a
        // difference), so the intervals tile [0, total) exactly.
        const int per = (nseg + 31) / 32;
        double run = 0.0;
        for (int s = lane * per; s < min(nseg, lane * per + per); ++s) run += (double)s_seg[s];
        double incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        double base = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) base = 0.0;
        for (int s = lane * per; s < min(nseg, lane * per + per); ++s) {
            base += (double)s_seg[s];
            s_segcum[s] = base;
        }
    }
    __syncthreads();
    if (tid == 0) s_res[2] = s_segcum[nseg - 1];  // CTA total
    __syncthreads();
    // cluster exclusive prefix of CTA totals
    if (tid == 0) s_red[parity] = RedSlot{s_res[2], 0.0, 0, 0};
    cluster.sync();
    if (warp == 0) {
        double tot = 0.0;
        if (lane < cs) tot = cluster.map_shared_rank(&s_red[parity], lane)->a;
        double incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        double excl = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) excl = 0.0;
        const double grand = __shfl_sync(0xffffffffu, incl, cs - 1);
        const double mine_incl = __shfl_sync(0xffffffffu, incl, rank);
        const double mine_excl = __shfl_sync(0xffffffffu, excl, rank);
        if (lane == 0) {
            const double target = (double)a.u_bonus[b] * grand;  // u in [0,1): target < grand
            s_res[0] = mine_excl;
            s_res[1] = target;
            s_ires[0] = (target >= mine_excl && target < mine_incl) ? 1 : 0;
        }
    }
    parity ^= 1;
    __syncthreads();
    if (s_ires[0]) {
        // this CTA holds the crossing: find the segment, then the lane, then the element
        const double target = s_res[1] - s_res[0];
        if (tid == 0) {
            int seg = -1;
            for (int s = 0; s < nseg; ++s)
                if (target < s_segcum[s]) {
                    seg = s;
                    break;
                }
            if (seg < 0)  // only by rounding of the base subtraction: last segment with mass
                for (int s = nseg - 1; s >= 0 && seg < 0; --s)
                    if (s_seg[s] > 0.0f) seg = s;
            s_ires[2] = seg;
            s_res[3] = target - (seg > 0 ? s_segcum[seg - 1] : 0.0);
        }
        __syncthreads();
        const int seg = s_ires[2];
        const int kseg = seg / nwarps, wseg = seg % nwarps;
        if (warp == wseg) {
            const float tgt = (float)s_res[3];
            float ts = 0.0f;
            float pe[4];
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if (k == kseg) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) pe[e] = pk[k][e];
                }
            ts = pe[0] + pe[1] + pe[2] + pe[3];
            float incl = ts;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.0f;
            const unsigned hit = __ballot_sync(0xffffffffu, tgt < incl && ts > 0.0f);
            const unsigned has = __ballot_sync(0xffffffffu, ts > 0.0f);
            // fp32 rounding can leave no lane past the target: take the last with mass
            const int l_sel = hit ? (__ffs(hit) - 1) : (31 - __clz(has));
            if (lane == l_sel) {
                float c = excl;
                int e_sel = -1, e_last = -1;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (pe[e] > 0.0f) e_last = e;
                    c += pe[e];
                    if (e_sel < 0 && tgt < c && pe[e] > 0.0f) e_sel = e;
                }
                if (e_sel < 0) e_sel = e_last;
                const int tok = v0 + (kseg * (int)blockDim.x + tid) * 4 + e_sel;
                a.bonus_token[b] = tok;
                a.out_tokens[rowoff + plen - 1] = tok;
            }
        }
    }
    cluster.sync();
}

}  // namespace tsv

namespace tsv {

template <int VEC, bool ALIGNED>
static cudaError_t launch_reject_inst(const SampleArgs& a, int B, int cs, int threads, cudaStream_t stream) {
    auto kern = tree_reject_kernel<VEC, ALIGNED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * cs), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Chooses the cluster size, block size and per-thread vector count for a vocabulary of
// V entries and B sequences, then launches one cluster per sequence.
cudaError_t launch_tree_reject(SampleArgs a, int B, int num_sms, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    const int V = a.V;
    int threads = 64;
    while (threads < 512 && threads * 4 * 2 < V) threads *= 2;
    const int cap1 = threads * 4 * 8;  // entries one CTA holds at VEC = 8
    int cs = 1;
    while (cs * cap1 < V) cs *= 2;  // smallest cluster that fits the row
    if (V > threads * 4 * 2) {      // rows long enough to be worth splitting further
        while (cs < 16 && B * cs * 2 <= 2 * num_sms) cs *= 2;
    }
    int vpc = (V + cs - 1) / cs;
    vpc = (vpc + 3) & ~3;
    a.v_per_cta = vpc;
    const int need = (vpc + threads * 4 - 1) / (threads * 4);
    const bool aligned = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0 &&
                         (a.probs == nullptr || (reinterpret_cast<uintptr_t>(a.probs) & 15) == 0);
    if (need <= 1) return aligned ? launch_reject_inst<1, true>(a, B, cs, threads, stream)
                                  : launch_reject_inst<1, false>(a, B, cs, threads, stream);
    if (need <= 2) return aligned ? launch_reject_inst<2, true>(a, B, cs, threads, stream)
                                  : launch_reject_inst<2, false>(a, B, cs, threads, stream);
    if (need <= 4) return aligned ? launch_reject_inst<4, true>(a, B, cs, threads, stream)
                                  : launch_reject_inst<4, false>(a, B, cs, threads, stream);
    if (need <= 8) return aligned ? launch_reject_inst<8, true>(a, B, cs, threads, stream)
                                  : launch_reject_inst<8, false>(a, B, cs, threads, stream);
    return cudaErrorInvalidValue;
}

}  // namespace tsv
