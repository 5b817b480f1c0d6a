// attn_tc.cu -- tree-masked paged attention on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM, K/V tiles staged by TMA), bf16 inputs.
//
// sglang report, "What is Tree-Attention?" and "Tree-based Speculative Decoding
// (EAGLE) Implementation Summary": all flattened tree tokens are verified in one
// pass; each sees the cached prefix (attention_mask) and its own ancestors,
// itself included (tree_attention_mask).
//
// One CTA = one work item (sequence b, kv head g, key chunk c, row group of up to
// 256 query rows = two M=128 tiles).  The query rows of a kv head are the N * Gq
// (node, head) pairs, so each K/V tile loaded from HBM feeds Gq * N rows.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: 128-key K and V tiles of the paged cache, one box per
//               (cache block, 64-wide half of D), 128B-swizzled, into a ring of slots;
//   warp 1      TMEM owner and MMA issuer: S_m = Q_m K^T (128 x 128, fp32 in TMEM) and
//               O_m += P_m V (128 x D, fp32 in TMEM), ping-ponging the two M tiles so
//               one tile's softmax overlaps the other tile's MMAs (with a single M tile,
//               S is double-buffered across key tiles instead);
//   warps 4-11  softmax, one thread per query row (warpgroup m owns M tile m): reads
//               its S row from TMEM, applies the prefix/ancestor mask, keeps a running
//               max (rescaling O in TMEM only when the max grows by more than 2^8) and
//               sum, writes P (bf16 pairs) back into TMEM over the S columns it has
//               read; the PV MMA takes P as its TMEM A operand, so shared memory holds
//               only Q and the K/V ring (5 slots of 128 keys at D = 128, two M tiles).
// Sequences whose prefix spans several chunks write (m, l, O / l) partials that the
// merge kernel combines; single-chunk sequences write the output directly.
// Every mbarrier wait is bounded (about one second); a timeout sets TSV_DERR_TIMEOUT
// for the sequence, lets the other roles drain, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {
namespace {

constexpr int kThreads = 384;
constexpr int kTileKeys = 128;
constexpr uint32_t kHalfBytes = 128 * 128;   // 128 rows x 64 bf16 (one 128B-swizzled half)
constexpr int kMaxSlots = 12;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ----------------------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Gives up after
// about one second, or at once when another role has already given up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]: A (M x K bf16) read from TMEM, lane = row,
// two K-consecutive elements per 32-bit column (lower half = lower k)
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrives on `bar` once every tcgen05 operation issued so far by this thread is complete
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

#define TSV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
// 32 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : TSV_R8(0), TSV_R8(8), TSV_R8(16), TSV_R8(24)
        : "r"(taddr));
}
#undef TSV_R8
#define TSV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        TSV_W8(0), TSV_W8(8), TSV_W8(16), TSV_W8(24)
        : "memory");
}
#undef TSV_W8
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory matrix descriptor, 128B swizzle, version 1 (tcgen05).
// lbo/sbo in bytes: K-major tiles use sbo = 1024 (8 rows x 128B) and no lbo; MN-major
// tiles use lbo = stride between 64-element column blocks and sbo = 1024.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// key t of the work item's range is visible to a row whose root-to-node path is the
// bit set anc: every prefix key (t < L) below the range end, and the tree key L + j iff
// node j is on the path
__device__ __forceinline__ bool key_visible(int t, int k_end, int L, uint32_t anc0, uint32_t anc1, uint32_t anc2,
                                            uint32_t anc3) {
    if (t >= k_end) return false;
    if (t < L) return true;
    const int jn = t - L;
    const uint32_t w = jn < 64 ? (jn < 32 ? anc0 : anc1) : (jn < 96 ? anc2 : anc3);
    return (w >> (jn & 31)) & 1u;
}

// byte offset of 16-byte chunk `q` (along the contiguous dimension) of row `row` in a
// tile stored as 64-element halves of [128 rows x 128 B], 128B-swizzled
__device__ __forceinline__ uint32_t sw128_offset(int row, int q) {
    const int half = q >> 3, cc = q & 7;
    return static_cast<uint32_t>(half * kHalfBytes + (row >> 3) * 1024 + (row & 7) * 128 + ((cc ^ (row & 7)) << 4));
}

struct TcLayout {
    uint32_t q0, ring, bars, misc, total;
    int slots;
};

template <int D>
__host__ __device__ inline TcLayout tc_layout(int nm_max) {
    // Q tiles (one per M tile) | ring of K/V slots | barriers | parents.  P lives in TMEM.
    TcLayout L{};
    const uint32_t qbytes = 128u * D * 2u, slot = 128u * D * 2u;
    L.q0 = 0;
    L.ring = (nm_max == 2 ? 2u : 1u) * qbytes;
    const uint32_t budget = 232448u - 1024u - 1024u;  // max dynamic smem - alignment slack - barriers/misc
    int slots = static_cast<int>((budget - L.ring) / slot);
    if (slots > kMaxSlots) slots = kMaxSlots;
    L.slots = slots;
    L.bars = L.ring + slots * slot;
    L.misc = L.bars + 512;
    L.total = L.misc + 512 + 1024;
    return L;
}

// barrier indices
struct Bars {
    static constexpr int kFull = 0;          // [slots]
    static constexpr int kEmpty = kMaxSlots;  // [slots]
    static constexpr int kS = 2 * kMaxSlots;  // [2]
    static constexpr int kP = kS + 2;         // [2]
    static constexpr int kO = kP + 2;         // [2]
    static constexpr int kQ = kO + 2;
    static constexpr int kDone = kQ + 1;
    static constexpr int kCount = kDone + 1;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   int nm_max) {
    constexpr int HALVES = D / 64;
    constexpr uint32_t SLOT = 128u * D * 2u;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const TcLayout lay = tc_layout<D>(nm_max);
    const int nslots = lay.slots;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    int* s_par = reinterpret_cast<int*>(smem + lay.misc);  // [128]
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + lay.bars + 8 * Bars::kCount);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + lay.bars + 8 * Bars::kCount + 4);
    int* s_flag = reinterpret_cast<int*>(smem + lay.bars + 8 * Bars::kCount + 8);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [=](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, g = blockIdx.y;
    const int mg = blockIdx.x % a.n_rgroups, c = blockIdx.x / a.n_rgroups;
    const int L = a.seq_lens[b];
    const int N = a.N;
    const int32_t* bt = a.block_table + (long long)b * a.max_blocks;

    // ---- validation (uniform).  Chunk-0 items check the whole sequence (they report
    // errors and poison rows); other chunks check only what they read.
    int e = 0;
    const int bs = 1 << a.bs_log2;
    if ((long long)L < 0 || (long long)L + N > (long long)a.max_blocks * bs) e = TSV_DERR_CAPACITY;
    const int nch = e ? 1 : num_chunks(L, a.chunk);
    if (c >= nch) return;
    const int k_begin = c * a.chunk;
    const int k_end = (c == nch - 1) ? L + N : min(L, (c + 1) * a.chunk);
    const bool has_tree = (c == nch - 1);
    if (c == 0 || has_tree) {
        if (!block_tree_ok(a.parent + (long long)b * N, N, s_flag)) e |= TSV_DERR_PARENT;
    }
    if (!(e & TSV_DERR_CAPACITY)) {
        const int blk0 = (c == 0) ? 0 : (k_begin >> a.bs_log2);
        const int blk1 = (c == 0) ? ((L + N + bs - 1) >> a.bs_log2) : ((k_end + bs - 1) >> a.bs_log2);
        if (tid == 0) *s_flag = 0;
        __syncthreads();
        for (int j = blk0 + tid; j < blk1; j += blockDim.x) {
            const int id = bt[j];
            if (id < 0 || id >= a.num_blocks) *s_flag = TSV_DERR_BLOCK;
        }
        __syncthreads();
        e |= *s_flag;
        __syncthreads();
    }
    const int r_base = mg * 256;
    const int nm = min(2, (a.R - r_base + 127) / 128);
    if (e) {
        if (c == 0) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
            const int r1 = min(a.R, r_base + 256);
            for (int idx = tid; idx < (r1 - r_base) * D; idx += blockDim.x) {
                const int r = r_base + idx / D, d = idx % D;
                const int n = r / a.G, h = g * a.G + r % a.G;
                out[(((long long)b * N + n) * a.Hq + h) * D + d] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
            }
            if (mg == 0 && g == 0 && tid == 0) a.seq_err[b] = e;
        }
        return;
    }
    if (c == 0 && mg == 0 && g == 0 && tid == 0) a.seq_err[b] = 0;
    const int ntiles = (k_end - k_begin + kTileKeys - 1) / kTileKeys;

    // ---- set-up: barriers, TMEM, parents
    if (tid == 0) {
        for (int i = 0; i < nslots; ++i) {
            mbar_init(bar(Bars::kFull + i), 1);
            mbar_init(bar(Bars::kEmpty + i), 1);
        }
        for (int m = 0; m < 2; ++m) {
            mbar_init(bar(Bars::kS + m), 1);
            mbar_init(bar(Bars::kP + m), 128);
            mbar_init(bar(Bars::kO + m), 1);
        }
        mbar_init(bar(Bars::kQ), 256);
        mbar_init(bar(Bars::kDone), 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), 512);
        tmem_relinquish();
    }
    if (has_tree)
        for (int i = tid; i < N; i += blockDim.x) s_par[i] = a.parent[(long long)b * N + i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    int my_err = 0;

    if (warp == 0) {
        // ============================ TMA producer (whole warp: lane j loads the id of
        // the tile's j-th cache block and issues that block's boxes, so a tile's block
        // ids are fetched in one coalesced load instead of one dependent load each)
        const int nfills = 2 * ntiles;
        // block id of this lane's cache block for fill f (K and V fills of a tile share ids);
        // loaded before waiting for the fill's slot so the load latency is hidden
        auto tile_block = [=](int f) -> int {
            const int t0 = k_begin + (f >> 1) * kTileKeys;
            const int nb = (min(t0 + kTileKeys, k_end) - t0 + bs - 1) >> a.bs_log2;
            return lane < nb ? bt[(t0 >> a.bs_log2) + lane] : 0;
        };
        int blk_next = tile_block(0);
        for (int f = 0; f < nfills && !my_err; ++f) {
            const int slot = f % nslots, use = f / nslots;
            const int blk = blk_next;
            if (f + 1 < nfills) blk_next = ((f + 1) >> 1) == (f >> 1) ? blk : tile_block(f + 1);
            if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(Bars::kEmpty + slot), (use - 1) & 1, s_abort))) {
                my_err = 1;
                break;
            }
            const int t0 = k_begin + (f >> 1) * kTileKeys;
            const int t1 = min(t0 + kTileKeys, k_end);
            const int nblk = (t1 - t0 + bs - 1) >> a.bs_log2;
            const CUtensorMap* map = (f & 1) ? &tmv : &tmk;
            const uint32_t dst = smem_u32(smem + lay.ring + slot * SLOT);
            if (lane == 0) mbar_expect_tx(bar(Bars::kFull + slot), static_cast<uint32_t>(nblk * bs * 128 * HALVES));
            __syncwarp();
            if (lane < nblk) {  // a 128-key tile spans at most 128 / 8 = 16 blocks
#pragma unroll
                for (int hh = 0; hh < HALVES; ++hh)
                    tma_load_3d(dst + hh * kHalfBytes + lane * bs * 128, map, bar(Bars::kFull + slot), hh * 64, g,
                                blk * bs);
            }
        }
        // never leave with copies in flight: wait for the latest fill of every slot
        if (lane == 0) {
            for (int f = max(0, 2 * ntiles - nslots); f < 2 * ntiles; ++f) {
                volatile int never = 0;
                if (!mbar_wait(bar(Bars::kFull + f % nslots), (f / nslots) & 1, &never)) my_err = 1;
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, 128, false);
            constexpr uint32_t idO = idesc_bf16(128, D, true);
            const uint32_t q_base = smem_u32(smem + lay.q0);
            const uint32_t ring_base = smem_u32(smem + lay.ring);
            // S buffer sb (TMEM columns sb*128) = Q tile qm . K^T
            auto issue_S = [=](int qm, int sb, int slot) {
                const uint32_t qa = q_base + qm * (128u * D * 2u);
                const uint32_t kb = ring_base + slot * SLOT;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
                    mma_bf16(tmem + sb * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), idS,
                             k > 0);
                }
            };
            // O tile om += P . V, P in TMEM over S buffer pb's columns (16 keys = 8 columns per MMA)
            auto issue_PV = [=](int om, int pb, int slot, bool acc_first) {
                const uint32_t vb = ring_base + slot * SLOT;
#pragma unroll
                for (int k = 0; k < kTileKeys / 16; ++k)
                    mma_bf16_ts(tmem + 256 + om * D, tmem + pb * 128 + k * 8,
                                sdesc_sw128(vb + k * 16 * 128, kHalfBytes, 1024), idO, (acc_first || k > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(bar(Bars::kQ), 0, s_abort);
            tc_fence_after();
            if (nm == 2) {
                // two M tiles ping-pong: one tile's softmax overlaps the other's MMAs
                ok = ok && mbar_wait(bar(Bars::kFull + 0), 0, s_abort);
                tc_fence_after();
                if (ok) {
                    for (int m = 0; m < nm; ++m) {
                        issue_S(m, m, 0);
                        mma_commit(bar(Bars::kS + m));
                    }
                    mma_commit(bar(Bars::kEmpty + 0));
                }
                for (int j = 0; j < ntiles && ok; ++j) {
                    const int fV = 2 * j + 1, fK = 2 * j + 2;
                    ok = mbar_wait(bar(Bars::kFull + fV % nslots), (fV / nslots) & 1, s_abort);
                    tc_fence_after();
                    for (int m = 0; m < nm && ok; ++m) {
                        ok = mbar_wait(bar(Bars::kP + m), j & 1, s_abort);
                        if (!ok) break;
                        tc_fence_after();
                        issue_PV(m, m, fV % nslots, j > 0);
                        mma_commit(bar(Bars::kO + m));
                        if (m == nm - 1) mma_commit(bar(Bars::kEmpty + fV % nslots));  // V_j's last reader issued
                        if (j + 1 < ntiles) {
                            if (m == 0) {
                                ok = mbar_wait(bar(Bars::kFull + fK % nslots), (fK / nslots) & 1, s_abort);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            issue_S(m, m, fK % nslots);
                            mma_commit(bar(Bars::kS + m));
                        }
                    }
                    if (!ok) break;
                    if (j + 1 < ntiles) mma_commit(bar(Bars::kEmpty + fK % nslots));
                }
            } else {
                // one M tile: S is double-buffered across key tiles (tile j in buffer j & 1),
                // so S(j+1) is computed while tile j's softmax runs.  K fills are consumed
                // ahead of V fills (K0, K1, V0, K2, V1, ...); the ring holds >= 3 slots.
                for (int jj = 0; jj < 2 && jj < ntiles && ok; ++jj) {
                    const int fK = 2 * jj;
                    ok = mbar_wait(bar(Bars::kFull + fK % nslots), (fK / nslots) & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_S(0, jj, fK % nslots);
                    mma_commit(bar(Bars::kS + jj));
                    mma_commit(bar(Bars::kEmpty + fK % nslots));
                }
                for (int j = 0; j < ntiles && ok; ++j) {
                    const int b2 = j & 1;
                    const int fV = 2 * j + 1, fK = 2 * j + 4;
                    ok = mbar_wait(bar(Bars::kFull + fV % nslots), (fV / nslots) & 1, s_abort) &&
                         mbar_wait(bar(Bars::kP + b2), (j >> 1) & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_PV(0, b2, fV % nslots, j > 0);
                    mma_commit(bar(Bars::kO + 0));
                    mma_commit(bar(Bars::kEmpty + fV % nslots));
                    if (j + 2 < ntiles) {
                        ok = mbar_wait(bar(Bars::kFull + fK % nslots), (fK / nslots) & 1, s_abort);
                        if (!ok) break;
                        tc_fence_after();
                        issue_S(0, b2, fK % nslots);  // after PV(j) has read P(j) from this buffer
                        mma_commit(bar(Bars::kS + b2));
                        mma_commit(bar(Bars::kEmpty + fK % nslots));
                    }
                }
            }
            if (!ok) my_err = 1;
            // drain: every issued MMA completes before TMEM is released
            mma_commit(bar(Bars::kDone));
            volatile int never = 0;
            if (!mbar_wait(bar(Bars::kDone), 0, &never)) my_err = 1;
        }
    } else if (warp >= 4) {
        // ============================ softmax warpgroups
        const int wg = (warp - 4) >> 2;
        const int tw = tid - 128 - wg * 128;  // TMEM lane = tile row handled by this thread
        // A partial M tile deals its rows round-robin over the four 32-lane quadrants of
        // TMEM (tile row tw holds row 4*(tw%32) + tw/32), so all four softmax warps share
        // the work; a full tile keeps the identity order.
        const int rows_here = min(128, a.R - r_base - wg * 128);
        const int rl = rows_here < 128 ? 4 * (tw & 31) + (tw >> 5) : tw;
        const int r = r_base + wg * 128 + rl;
        const bool valid = (wg < nm) && (rl < rows_here);
        const int n = valid ? r / a.G : 0;
        const int h = g * a.G + (valid ? r % a.G : 0);
        // Q row -> swizzled shared tile
        {
            uint8_t* qt = smem + lay.q0 + wg * (128u * D * 2u);
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                              (((long long)b * N + n) * a.Hq + h) * D);
            if (wg < nm) {
#pragma unroll
                for (int qq = 0; qq < D / 8; ++qq) {
                    uint4 v = valid ? __ldg(src + qq) : make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(qt + sw128_offset(tw, qq)) = v;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(Bars::kQ));
        }
        // ancestor mask of this row's node (tree keys only)
        uint32_t anc0 = 0u, anc1 = 0u, anc2 = 0u, anc3 = 0u;
        if (valid && has_tree) {
            int x = n;
            for (int step = 0; step <= N && x >= 0 && x < N; ++step) {
                const uint32_t bit = 1u << (x & 31);
                const int w = x >> 5;
                anc0 |= w == 0 ? bit : 0u;
                anc1 |= w == 1 ? bit : 0u;
                anc2 |= w == 2 ? bit : 0u;
                anc3 |= w == 3 ? bit : 0u;
                x = s_par[x];
            }
        }
        const bool warp_active = __any_sync(0xffffffffu, valid) && (wg < nm);
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS0 = tmem + lane_base;
        const uint32_t tO = tmem + lane_base + 256 + wg * D;
        float m_run = -INFINITY, l_run = 0.0f;
        const float sl2 = a.scale_log2;
        bool ok = true;
        for (int j = 0; j < ntiles && wg < nm; ++j) {
            const int t0 = k_begin + j * kTileKeys;
            // S/P buffer of this tile: the warpgroup's own with two M tiles; alternating
            // buffers (double-buffered S) with one
            const int sb = nm == 2 ? wg : (j & 1);
            const uint32_t sphase = nm == 2 ? (j & 1) : ((j >> 1) & 1);
            const uint32_t tS = tS0 + sb * 128;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bars::kS + sb), sphase, s_abort));
            if (!ok) break;
            tc_fence_after();
            if (warp_active) {
                // Two passes over the S row in TMEM, 64 columns per wait: the raw max
                // first, then P = 2^(s*scale - m) written as bf16 into the swizzled P
                // tile.  Independent accumulators (8 for the max, 4 for the sum) keep the
                // FMNMX/MUFU latency chains short; the masked path is taken only for
                // tiles that reach past the prefix.
                const bool full_tile = (t0 + kTileKeys <= L) && (t0 + kTileKeys <= k_end);
                float mxa[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxa[i] = -INFINITY;
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t pa[32], pb[32];
                    tmem_ld32(tS + h2 * 64, pa);
                    tmem_ld32(tS + h2 * 64 + 32, pb);
                    tmem_wait_ld();
                    if (valid) {
                        if (full_tile) {
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc) {
                                mxa[cc & 7] = fmaxf(mxa[cc & 7], __uint_as_float(pa[cc]));
                                mxa[cc & 7] = fmaxf(mxa[cc & 7], __uint_as_float(pb[cc]));
                            }
                        } else {
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc) {
                                const int c0 = h2 * 64 + cc;
                                if (key_visible(t0 + c0, k_end, L, anc0, anc1, anc2, anc3))
                                    mxa[cc & 7] = fmaxf(mxa[cc & 7], __uint_as_float(pa[cc]));
                                if (key_visible(t0 + c0 + 32, k_end, L, anc0, anc1, anc2, anc3))
                                    mxa[cc & 7] = fmaxf(mxa[cc & 7], __uint_as_float(pb[cc]));
                            }
                        }
                    }
                }
                const float mx_raw = fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
                                           fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
                const float mx = mx_raw * sl2;  // scale > 0: max commutes with it
                // the PV product of the previous tile must be done before O or P change
                if (j > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(Bars::kO + wg), (j - 1) & 1, s_abort));
                    tc_fence_after();
                }
                const float m_new = fmaxf(m_run, mx);
                bool rescale = false;
                float factor = 1.0f;
                if (m_run == -INFINITY) {
                    m_run = m_new;
                } else if (m_new > m_run + 8.0f) {
                    factor = ex2(m_run - m_new);
                    m_run = m_new;
                    rescale = true;
                }
                l_run *= factor;
                if (__any_sync(0xffffffffu, rescale) && ok) {
#pragma unroll 1
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t ov[32];
                        tmem_ld32(tO + q4 * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) ov[cc] = __float_as_uint(__uint_as_float(ov[cc]) * factor);
                        tmem_st32(tO + q4 * 32, ov);
                    }
                    tmem_wait_st();
                }
                const bool live = valid && m_run != -INFINITY;
                const float neg_m = -m_run;
                float la[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t pa[32], pb[32];
                    tmem_ld32(tS + h2 * 64, pa);
                    tmem_ld32(tS + h2 * 64 + 32, pb);
                    tmem_wait_ld();
                    // P in place of the scores (as bit patterns): pa = columns 0..31, pb = 32..63
                    if (live && full_tile) {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) {
                            pa[cc] = __float_as_uint(ex2(fmaf(__uint_as_float(pa[cc]), sl2, neg_m)));
                            pb[cc] = __float_as_uint(ex2(fmaf(__uint_as_float(pb[cc]), sl2, neg_m)));
                        }
                    } else if (live) {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) {
                            const int c0 = h2 * 64 + cc;
                            pa[cc] = key_visible(t0 + c0, k_end, L, anc0, anc1, anc2, anc3)
                                         ? __float_as_uint(ex2(fmaf(__uint_as_float(pa[cc]), sl2, neg_m)))
                                         : 0u;
                            pb[cc] = key_visible(t0 + c0 + 32, k_end, L, anc0, anc1, anc2, anc3)
                                         ? __float_as_uint(ex2(fmaf(__uint_as_float(pb[cc]), sl2, neg_m)))
                                         : 0u;
                        }
                    } else {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) pa[cc] = pb[cc] = 0u;
                    }
                    // pack to bf16 pairs and store over the S columns already read
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float p0 = __uint_as_float(i < 16 ? pa[2 * i] : pb[2 * i - 32]);
                        const float p1 = __uint_as_float(i < 16 ? pa[2 * i + 1] : pb[2 * i - 31]);
                        la[i & 3] += p0 + p1;
                        __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
                        w[i] = *reinterpret_cast<uint32_t*>(&pk);
                    }
                    tmem_st32(tS + h2 * 32, w);
                }
                tmem_wait_st();
                l_run += (la[0] + la[1]) + (la[2] + la[3]);
            }
            // the last tile's V rows past the key range are zeroed before the PV product
            // (they may hold stale or foreign data; P is 0 there but 0 * NaN is NaN)
            if (wg == 0 && j == ntiles - 1 && k_end - t0 < kTileKeys) {
                const int fV = 2 * j + 1;
                ok = ok && mbar_wait(bar(Bars::kFull + fV % nslots), (fV / nslots) & 1, s_abort);
                if (ok) {
                    uint8_t* vt = smem + lay.ring + (fV % nslots) * SLOT;
                    const int row0 = k_end - t0;
                    const int nbytes_row = 128;
                    for (int idx = tw; idx < (kTileKeys - row0) * HALVES * (nbytes_row / 16); idx += 128) {
                        const int per_half = (kTileKeys - row0) * 8;
                        const int hh = idx / per_half, rem = idx % per_half;
                        const int row = row0 + rem / 8, cq = rem % 8;
                        *reinterpret_cast<uint4*>(vt + hh * kHalfBytes + row * 128 + cq * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            fence_proxy_async_smem();  // the zeroed V rows, written through the generic proxy
            tc_fence_before();
            mbar_arrive(bar(Bars::kP + sb));
            if (!ok) break;
        }
        // epilogue: O / l
        if (ok && wg < nm && ntiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bars::kO + wg), (ntiles - 1) & 1, s_abort));
            tc_fence_after();
        }
        if (ok && warp_active) {
            const float inv = 1.0f / l_run;
            const long long orow = (((long long)b * N + n) * a.Hq + h) * D;
            const long long prow = (((long long)b * a.Hkv + g) * a.max_chunks + c) * a.R + r;
#pragma unroll
            for (int q4 = 0; q4 < D / 32; ++q4) {
                uint32_t ov[32];
                tmem_ld32(tO + q4 * 32, ov);
                tmem_wait_ld();
                if (valid) {
                    if (nch == 1) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + q4 * 32);
#pragma unroll
                        for (int v8 = 0; v8 < 4; ++v8) {
                            uint32_t w[4];
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) {
                                __nv_bfloat162 pk = __floats2bfloat162_rn(__uint_as_float(ov[v8 * 8 + 2 * e2]) * inv,
                                                                          __uint_as_float(ov[v8 * 8 + 2 * e2 + 1]) * inv);
                                w[e2] = *reinterpret_cast<uint32_t*>(&pk);
                            }
                            dst[v8] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(a.part_o + prow * D + q4 * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(__uint_as_float(ov[v4 * 4]) * inv, __uint_as_float(ov[v4 * 4 + 1]) * inv,
                                                  __uint_as_float(ov[v4 * 4 + 2]) * inv,
                                                  __uint_as_float(ov[v4 * 4 + 3]) * inv);
                    }
                }
            }
            if (valid && nch > 1) {
                a.part_m[prow] = m_run;
                a.part_l[prow] = l_run;
            }
        }
        if (!ok) my_err = 1;
    }
    if (my_err) {
        *s_abort = 1;
        atomicOr(&a.seq_err[b], TSV_DERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D view of a [num_blocks * bs, Hkv, D] bf16 cache: box = 64 head dims x 1 kv head x bs slots
bool make_cache_map(CUtensorMap* map, const void* base, int D, int Hkv, long long rows, int bs) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hkv) * D * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(bs)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc_inst(const AttnArgs& a, cudaStream_t stream) {
    CUtensorMap mk, mv;
    const long long rows = static_cast<long long>(a.num_blocks) << a.bs_log2;
    if (!make_cache_map(&mk, a.k_cache, D, a.Hkv, rows, 1 << a.bs_log2) ||
        !make_cache_map(&mv, a.v_cache, D, a.Hkv, rows, 1 << a.bs_log2))
        return cudaErrorInvalidValue;
    const int nm_max = a.R > 128 ? 2 : 1;
    const TcLayout lay = tc_layout<D>(nm_max);
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(lay.total));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(a.n_rgroups * a.max_chunks), static_cast<unsigned>(a.Hkv),
              static_cast<unsigned>(a.B));
    attn_tc_kernel<D><<<grid, kThreads, lay.total, stream>>>(a, mk, mv, nm_max);
    return cudaGetLastError();
}

}  // namespace

bool attn_tc_supported(int D) { return D == 64 || D == 128; }
int attn_tc_rows_per_cta() { return 256; }

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream) {
    return a.D == 64 ? launch_tc_inst<64>(a, stream) : launch_tc_inst<128>(a, stream);
}

}  // namespace tsv
