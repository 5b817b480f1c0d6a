// attn_simt.cu -- tree-masked attention on the FMA pipes (fp32 inputs), and the
// split-K merge shared with the tensor-core path (bf16 inputs).
//
// sglang report, "What is Tree-Attention?" and "Tree-based Speculative Decoding
// (EAGLE) Implementation Summary": the flattened tree's tokens are scored in one
// pass; each tree node sees the cached prefix and its own ancestors (itself
// included) among the tree tokens.
//
// fp32 inputs stay on FFMA: a TF32 tensor-core product would not meet a 1e-4
// error bound.  Each work item stages 32-key K/V tiles of one kv head in shared
// memory (converted to fp32) and each warp runs an online softmax for its query
// rows: lane = key for the scores, lane = head dimension for the output.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {

constexpr int kSimtRows = 16;   // rows per work item (2 per warp)
constexpr int kSimtTile = 32;   // keys per shared-memory tile
constexpr int kSimtThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Per-sequence validation shared by all attention kernels: tree shape, capacity and
// block ids.  Returns the TSV_DERR_* bits (same precedence as the definition).
__device__ __forceinline__ int attn_validate(const AttnArgs& a, int b, int* s_flag) {
    int e = block_tree_ok(a.parent + (long long)b * a.N, a.N, s_flag) ? 0 : TSV_DERR_PARENT;
    e |= block_cache_errors(a.block_table + (long long)b * a.max_blocks, a.seq_lens[b], a.N, 1 << a.bs_log2,
                            a.max_blocks, a.num_blocks, s_flag);
    return e;
}

// Writes NaN into the rows [r0, r1) of (b, kv head g) of the output.
template <typename T>
__device__ __forceinline__ void attn_poison_rows(const AttnArgs& a, int b, int g, int r0, int r1) {
    T* out = static_cast<T*>(a.out);
    const int D = a.D;
    for (int idx = threadIdx.x; idx < (r1 - r0) * D; idx += blockDim.x) {
        const int r = r0 + idx / D, d = idx % D;
        const int n = r / a.G, h = g * a.G + r % a.G;
        out[(((long long)b * a.N + n) * a.Hq + h) * D + d] = from_f32<T>(__int_as_float(0x7fc00000));
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads) attn_simt_kernel(const AttnArgs a) {
    constexpr int DP = D / 32;  // output dims per lane
    __shared__ float s_q[kSimtRows][D];
    __shared__ float s_k[kSimtTile][D + 1];
    __shared__ float s_v[kSimtTile][D];
    __shared__ uint32_t s_anc[kMaxNodes][4];
    __shared__ int s_flag;

    const int b = blockIdx.z, g = blockIdx.y;
    const int rg = blockIdx.x % a.n_rgroups, c = blockIdx.x / a.n_rgroups;
    const int L = a.seq_lens[b];
    const int e = attn_validate(a, b, &s_flag);
    const int nch = e ? 1 : num_chunks(L, a.chunk);
    if (c >= nch) return;
    const int r0 = rg * kSimtRows, r1 = min(a.R, r0 + kSimtRows);
    if (e) {
        if (c == 0) attn_poison_rows<T>(a, b, g, r0, r1);
        if (c == 0 && rg == 0 && g == 0 && threadIdx.x == 0) a.seq_err[b] = e;
        return;
    }
    if (c == 0 && rg == 0 && g == 0 && threadIdx.x == 0) a.seq_err[b] = 0;

    const int32_t* par = a.parent + (long long)b * a.N;
    const int32_t* bt = a.block_table + (long long)b * a.max_blocks;
    build_ancestor_masks(par, a.N, s_anc);
    const T* q = static_cast<const T*>(a.q);
    for (int idx = threadIdx.x; idx < kSimtRows * D; idx += blockDim.x) {
        const int rr = idx / D, d = idx % D, r = r0 + rr;
        float v = 0.0f;
        if (r < r1) {
            const int n = r / a.G, h = g * a.G + r % a.G;
            v = to_f32<T>(q[(((long long)b * a.N + n) * a.Hq + h) * D + d]);
        }
        s_q[rr][d] = v;
    }
    const int k_begin = c * a.chunk;
    const int k_end = (c == nch - 1) ? L + a.N : min(L, (c + 1) * a.chunk);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float m[2], l[2], o[2][DP];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < DP; ++j) o[i][j] = 0.0f;
    }
    const T* kc = static_cast<const T*>(a.k_cache);
    const T* vc = static_cast<const T*>(a.v_cache);
    for (int t0 = k_begin; t0 < k_end; t0 += kSimtTile) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kSimtTile * D; idx += blockDim.x) {
            const int kk = idx / D, d = idx % D, t = t0 + kk;
            float kv = 0.0f, vv = 0.0f;
            if (t < k_end) {
                const long long off = (phys_row(bt, t, a.bs_log2) * a.Hkv + g) * D + d;
                kv = to_f32<T>(kc[off]);
                vv = to_f32<T>(vc[off]);
            }
            s_k[kk][d] = kv;
            s_v[kk][d] = vv;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rr = warp * 2 + i, r = r0 + rr;
            if (r >= r1) continue;
            const int n = r / a.G;
            const int t = t0 + lane;
            bool vis = t < k_end;
            if (vis && t >= L) vis = anc_has(s_anc[n], t - L);
            float s = -INFINITY;
            if (vis) {
                float acc = 0.0f;
#pragma unroll 8
                for (int d = 0; d < D; ++d) acc = fmaf(s_q[rr][d], s_k[lane][d], acc);
                s = acc * a.scale_log2;
            }
            float tmax = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float mnew = fmaxf(m[i], tmax);
            if (mnew == -INFINITY) continue;  // nothing visible yet
            const float corr = exp2f(m[i] - mnew);
            const float p = vis ? exp2f(s - mnew) : 0.0f;
            float psum = p;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l[i] = l[i] * corr + psum;
            m[i] = mnew;
#pragma unroll
            for (int j = 0; j < DP; ++j) o[i][j] *= corr;
            for (int kk = 0; kk < kSimtTile; ++kk) {
                const float pk = __shfl_sync(0xffffffffu, p, kk);
                if (pk != 0.0f) {
#pragma unroll
                    for (int j = 0; j < DP; ++j) o[i][j] = fmaf(pk, s_v[kk][lane + 32 * j], o[i][j]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int rr = warp * 2 + i, r = r0 + rr;
        if (r >= r1) continue;
        const int n = r / a.G, h = g * a.G + r % a.G;
        const float inv = 1.0f / l[i];
        if (nch == 1) {
            T* out = static_cast<T*>(a.out);
#pragma unroll
            for (int j = 0; j < DP; ++j)
                out[(((long long)b * a.N + n) * a.Hq + h) * D + lane + 32 * j] = from_f32<T>(o[i][j] * inv);
        } else {
            const long long prow = (((long long)b * a.Hkv + g) * a.max_chunks + c) * a.R + r;
#pragma unroll
            for (int j = 0; j < DP; ++j) a.part_o[prow * D + lane + 32 * j] = o[i][j] * inv;
            if (lane == 0) {
                a.part_m[prow] = m[i];
                a.part_l[prow] = l[i];
            }
        }
    }
}

// Combines the chunk partials of every multi-chunk sequence: with M = max_s m_s,
// out = sum_s 2^(m_s - M) l_s O_s / sum_s 2^(m_s - M) l_s  (m in log2 units).
// One warp per (b, n, h) row; lane = head dimension.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnArgs a) {
    constexpr int DP = D / 32;
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)a.B * a.N * a.Hq) return;
    const int h = (int)(row % a.Hq);
    const int n = (int)((row / a.Hq) % a.N);
    const int b = (int)(row / ((long long)a.Hq * a.N));
    if (a.seq_err[b]) return;
    const int nch = num_chunks(a.seq_lens[b], a.chunk);
    if (nch == 1) return;
    const int g = h / a.G, r = n * a.G + h % a.G;
    const long long base = (((long long)b * a.Hkv + g) * a.max_chunks) * a.R + r;
    float M = -INFINITY;
    for (int s = lane; s < nch; s += 32) M = fmaxf(M, a.part_m[base + (long long)s * a.R]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[DP];
#pragma unroll
    for (int j = 0; j < DP; ++j) acc[j] = 0.0f;
    float wsum = 0.0f;
    for (int s = 0; s < nch; ++s) {
        const long long pr = base + (long long)s * a.R;
        const float w = a.part_l[pr] * exp2f(a.part_m[pr] - M);
        wsum += w;
#pragma unroll
        for (int j = 0; j < DP; ++j) acc[j] = fmaf(w, a.part_o[pr * D + lane + 32 * j], acc[j]);
    }
    const float inv = 1.0f / wsum;
    T* out = static_cast<T*>(a.out);
#pragma unroll
    for (int j = 0; j < DP; ++j) out[row * D + lane + 32 * j] = from_f32<T>(acc[j] * inv);
}

template <int D>
static cudaError_t launch_simt_inst(const AttnArgs& a, cudaStream_t stream) {
    dim3 grid((unsigned)(a.n_rgroups * a.max_chunks), (unsigned)a.Hkv, (unsigned)a.B);
    attn_simt_kernel<float, D><<<grid, kSimtThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// Fused append on the FMA path: one CTA per sequence writes the tree's rows where the
// capacity and block ids allow it (the attention kernel after it in the stream checks
// and reports the sequence).
__global__ void __launch_bounds__(128) attn_append_kernel(const AttnArgs a) {
    __shared__ int s_flag;
    const int b = blockIdx.x;
    const int L = a.seq_lens[b];
    const int32_t* bt = a.block_table + (long long)b * a.max_blocks;
    if (block_cache_errors(bt, L, a.N, 1 << a.bs_log2, a.max_blocks, a.num_blocks, &s_flag)) return;
    append_tree_rows(a.k_new, a.v_new, a.k_cache_w, a.v_cache_w, bt, b, L, a.N, a.Hkv * a.D * 4, a.bs_log2,
                     ((long long)a.num_blocks << a.bs_log2) * a.Hkv * a.D * 4 / 16,
                     (long long)a.B * a.N * a.Hkv * a.D * 4 / 16, a.seq_err + b);
}

// fp32 inputs only: bf16 runs on the tensor-core kernel (attn_tc.cu)
cudaError_t launch_attn_simt_f32(const AttnArgs& a, cudaStream_t stream) {
    if (a.k_new != nullptr) {
        attn_append_kernel<<<a.B, 128, 0, stream>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return a.D == 64 ? launch_simt_inst<64>(a, stream) : launch_simt_inst<128>(a, stream);
}

template <typename T, int D>
static cudaError_t launch_merge_inst(const AttnArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.B * a.N * a.Hq;
    attn_merge_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attn_merge(const AttnArgs& a, bool bf16, cudaStream_t stream) {
    if (a.max_chunks == 1) return cudaSuccess;
    if (bf16) return a.D == 64 ? launch_merge_inst<__nv_bfloat16, 64>(a, stream)
                               : launch_merge_inst<__nv_bfloat16, 128>(a, stream);
    return a.D == 64 ? launch_merge_inst<float, 64>(a, stream) : launch_merge_inst<float, 128>(a, stream);
}

}  // namespace tsv
