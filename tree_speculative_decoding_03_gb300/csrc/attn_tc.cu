// attn_tc.cu -- tree-masked paged attention on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM, K/V tiles staged by TMA), bf16 inputs.
//
// sglang report, "What is Tree-Attention?" and "Tree-based Speculative Decoding
// (EAGLE) Implementation Summary": all flattened tree tokens are verified in one
// pass; each sees the cached prefix (attention_mask) and its own ancestors,
// itself included (tree_attention_mask).
//
// Work split (persistent, stream-K style): the keys [0, L_b + N) of every unit
// (sequence b, kv head g) are cut into 128-key tiles; the tiles of all units, b-major,
// form one sequence that is cut evenly between `lanes` CTAs per row group, so every CTA
// streams the same number of K/V tiles whatever the mix of prefix lengths.  The CTA of
// row group rg handles query rows [256 rg, 256 rg + 256) of each unit (up to two M=128
// tiles).  The query rows of a unit are the N * Gq (node, head) pairs, so each K/V tile
// loaded from HBM feeds Gq * N rows.  A CTA walks its tiles as segments, one per unit
// it touches; a segment that covers its whole unit writes the output directly, the
// others write (m, l, O / l) partials to a per-CTA slot, which a merge kernel over all
// SMs combines (log-sum-exp).  A small kernel checks every sequence (seq_err) while the
// attention runs: the schedule depends only on the lengths, a flagged sequence's tiles
// are computed anyway (reads stay inside the cache: out-of-range tensor-map boxes read
// zeros) and the merge kernel, which runs after both, writes its rows as NaN.  The
// kernels are chained with programmatic dependent launch.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: 128-key K and V tiles of the paged cache, one box per
//               (cache block, 64-wide half of D), 128B-swizzled, into a ring of slots,
//               running ahead across segment boundaries;
//   warp 1      TMEM owner and MMA issuer: S_m = Q_m K^T (128 x 128, fp32 in TMEM) and
//               O_m += P_m V (128 x D, fp32 in TMEM), ping-ponging the two M tiles so
//               one tile's softmax overlaps the other tile's MMAs (with a single M tile,
//               S is double-buffered across key tiles instead);
//   warp 2      (set-up only) locates this CTA's first tile;
//   warps 4-11  softmax, one thread per query row (warpgroup m owns M tile m): loads
//               the segment's Q rows, reads its S row from TMEM, applies the prefix /
//               ancestor mask, keeps a running max (rescaling O in TMEM only when the
//               max grows by more than 2^8) and sum, writes P (bf16 pairs) back into
//               TMEM over the S columns it has read; the PV MMA takes P as its TMEM A
//               operand, so shared memory holds only Q and the K/V ring.
// Every mbarrier wait is bounded (about one second); a timeout sets TSV_DERR_TIMEOUT
// for the sequence being worked on, lets the other roles drain, frees TMEM and returns.
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
#ifdef TSV_TEST_HOOKS
// test build only: waits give up after 1 ms, and one wait can be pointed at a barrier
// that nothing completes (tsv_test_set_stall), so a test can drive the timeout path
constexpr unsigned long long kWaitLimitNs = 1000000ull;
__device__ int g_test_stall = 0;
#else
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
#endif
// A CTA with few tiles sends its first K/V tile out alone and waits for the K half before
// filling the rest of the ring: at start-up every such CTA's first tile then sits at the
// front of the DRAM queue instead of behind every CTA's whole ring (measured: chain5
// 42.6 -> 41.6 us; with long runs the start-up does not matter and it is skipped).
constexpr int kFirstTileAloneMaxTiles = 16;

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
// L2 policy for data read once: its lines are the first to be evicted, so the stream of
// K/V tiles does not push out the code, Q rows, parents and block tables that every CTA
// reads at its unit boundaries (measured: 1 - 3 % less time per launch)
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
        "%4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
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
// three-input maximum (one instruction on sm_100 and later)
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// packed pairs of fp32 (one instruction per pair on sm_100 and later)
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// register budget per thread after the set-up: the producer / MMA warpgroup gives up
// registers, the softmax warpgroups (which hold a whole 128-key S row) take them:
// 128 x 96 + 256 x 200 <= 384 x 168, the registers the CTA is launched with
template <uint32_t R>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R)); }
template <uint32_t R>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R)); }
constexpr uint32_t kRegsProducer = 96, kRegsSoftmax = 200;
static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= 384 * 168, "register split exceeds the launch");

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

// Visibility of 32 consecutive keys to a row whose root-to-node path is the bit set
// anc (bits 0..N-1 only): bit c covers the key with tree index base + c, i.e. key
// L + base + c.  Every prefix key (tree index < 0) is visible, and the tree key L + j
// iff node j is on the path; keys past the last node have no bit in anc, so they are
// hidden too.
__device__ __forceinline__ uint32_t vis_word(int base, uint32_t anc0, uint32_t anc1, uint32_t anc2,
                                             uint32_t anc3) {
    if (base <= -32) return 0xffffffffu;
    if (base >= 128) return 0u;
    if (base < 0) return (0xffffffffu >> (32 + base)) | (anc0 << -base);
    const int wi = base >> 5;
    const uint32_t lo = wi == 0 ? anc0 : (wi == 1 ? anc1 : (wi == 2 ? anc2 : anc3));
    const uint32_t hi = wi == 0 ? anc1 : (wi == 1 ? anc2 : (wi == 2 ? anc3 : 0u));
    return __funnelshift_r(lo, hi, static_cast<uint32_t>(base & 31));
}

// 16-byte global -> shared copy completing asynchronously (zero-filled when !take)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool take) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(take ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ uint32_t opaque_u32(uint32_t x) {
    uint32_t y;
    asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

struct TcLayout {
    uint32_t q0, ring, bars, misc, total;
    int slots;
};

template <int D>
__host__ __device__ inline TcLayout tc_layout(int nm_max) {
    // Q tiles (one per M tile) | ring of K/V slots | barriers | misc.  P lives in TMEM.
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
    static constexpr int kQ = kO + 2;         // one phase per segment
    static constexpr int kDone = kQ + 1;
    static constexpr int kStall = kDone + 1;  // never completed (test build: the stalled wait)
    static constexpr int kCount = kStall + 1;
};

// misc region (512 bytes): parents of the segment's sequence (int8, two buffers by
// segment parity), per-slot fill metadata, the CTA's schedule, the first tile's block ids
constexpr uint32_t kMiscPar = 0, kMiscMeta = 256, kMiscSched = 320, kMiscBlk0 = 384;

// Tiles of each unit of sequence b: 0 when its length does not fit the block table
// (so no block-table entry past the row is read), else ceil((L_b + N) / 128).  It depends
// on the lengths only, so it needs nothing from the check kernel running alongside.
__device__ __forceinline__ int seq_tiles(const AttnArgs& a, int b, int* L_out) {
    const int L = __ldg(a.seq_lens + b);
    *L_out = L;
    if (L < 0 || (long long)L + a.N > ((long long)a.max_blocks << a.bs_log2)) return 0;
    return (L + a.N + kTileKeys - 1) / kTileKeys;
}

// Position in a CTA's run of tiles: unit (b, g), tile t of its Tb tiles, prefix L.
struct TileIt {
    int b, g, t, Tb, L;
    // first tile of the next unit that has tiles (sequences without tiles are skipped)
    __device__ __forceinline__ void next_unit(const AttnArgs& a) {
        t = 0;
        if (++g < a.Hkv) return;
        g = 0;
        do {
            ++b;
            Tb = b < a.B ? seq_tiles(a, b, &L) : 1;
        } while (b < a.B && Tb == 0);
    }
    __device__ __forceinline__ void next(const AttnArgs& a) {
        if (t + 1 < Tb)
            ++t;
        else
            next_unit(a);
    }
};

// lane owning global tile x when T tiles are cut into `lanes` runs [k T / lanes, (k+1) T / lanes)
__device__ __forceinline__ int lane_of_tile(long long x, long long T, int lanes) {
    return static_cast<int>(((x + 1) * lanes - 1) / T);
}
__device__ __forceinline__ long long lane_start(int k, long long T, int lanes) { return (long long)k * T / lanes; }

// One warp: total tiles, this lane's run [s, e), the unit/tile where it starts and
// the block ids of that first tile (so the first copies need no global read after the
// set-up barrier).  sched: b, g, t, Tb, L, count, s (2 words), T (2 words);
// blk0[j] = id of the first tile's j-th cache block (j < 16).
__device__ __forceinline__ void find_start(const AttnArgs& a, int lane_c, int* sched, int* blk0) {
    const int lane = threadIdx.x & 31;
    long long T = 0;
    int tb_first = 0, L_first = 0;  // the first 32 sequences, kept for the second pass
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        int L = 0;
        const int b = b0 + lane;
        const int tb = b < a.B ? seq_tiles(a, b, &L) : 0;
        if (b0 == 0) {
            tb_first = tb;
            L_first = L;
        }
        T += tb;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) T += __shfl_xor_sync(0xffffffffu, T, o);
    T *= a.Hkv;
    const long long s = lane_start(lane_c, T, a.lanes), e = lane_start(lane_c + 1, T, a.lanes);
    int fb = 0, fg = 0, ft = 0, fTb = 1, fL = 0;
    if (e > s) {
        long long base = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            int L = L_first;
            const int b = b0 + lane;
            const int tb = b0 == 0 ? tb_first : (b < a.B ? seq_tiles(a, b, &L) : 0);
            const long long w = (long long)tb * a.Hkv;
            long long incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const long long excl = incl - w;
            const unsigned hit = __ballot_sync(0xffffffffu, w > 0 && base + excl <= s && s < base + incl);
            if (hit) {
                const int src = __ffs(hit) - 1;
                const long long off = s - (base + excl);
                const int mg = static_cast<int>(off / (tb > 0 ? tb : 1)), mt = static_cast<int>(off % (tb > 0 ? tb : 1));
                fb = __shfl_sync(0xffffffffu, b, src);
                fg = __shfl_sync(0xffffffffu, mg, src);
                ft = __shfl_sync(0xffffffffu, mt, src);
                fTb = __shfl_sync(0xffffffffu, tb, src);
                fL = __shfl_sync(0xffffffffu, L, src);
                break;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    if (lane == 0) {
        sched[0] = fb;
        sched[1] = fg;
        sched[2] = ft;
        sched[3] = fTb;
        sched[4] = fL;
        sched[5] = static_cast<int>(e - s);
        reinterpret_cast<long long*>(sched)[3] = s;  // words 6-7
        reinterpret_cast<long long*>(sched)[4] = T;  // words 8-9
    }
    if (e > s && lane < 16) {
        const int u0 = ft * kTileKeys;
        const int nb = (min(u0 + kTileKeys, fL + a.N) - u0 + (1 << a.bs_log2) - 1) >> a.bs_log2;
        blk0[lane] = lane < nb ? __ldg(a.block_table + (long long)fb * a.max_blocks + (u0 >> a.bs_log2) + lane) : 0;
    }
}

// One CTA per sequence, alongside the attention kernel: the checks behind seq_err[b]
// (capacity first; a parent array that is not a tree; a block id outside the cache),
// and with the fused append the tree's new K/V rows (256 threads then, 128 without).
__global__ void __launch_bounds__(256) attn_tc_check_kernel(const AttnArgs a) {
    __shared__ int s_flag;
    // the inputs may come from the previous kernel in the stream: wait for it before the
    // attention kernel (which reads them too) is allowed to start
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x, N = a.N;
    const int L = a.seq_lens[b];
    const bool cap_ok = L >= 0 && (long long)L + N <= ((long long)a.max_blocks << a.bs_log2);
    int e = cap_ok ? 0 : TSV_DERR_CAPACITY;
    if (!block_tree_ok(a.parent + (long long)b * N, N, &s_flag)) e |= TSV_DERR_PARENT;
    if (cap_ok)
        e |= block_cache_errors(a.block_table + (long long)b * a.max_blocks, L, N, 1 << a.bs_log2, a.max_blocks,
                                a.num_blocks, &s_flag);
    // fused append: the tree's rows go into the cache here, where the block ids have just
    // been checked; the attention kernel waits for this kernel before its first tile
    // that reaches the tree keys
    if (threadIdx.x == 0) a.seq_err[b] = e;
    __syncthreads();  // the checked build's index checks may add a bit to it below
    if (a.k_new != nullptr && cap_ok && !(e & TSV_DERR_BLOCK))
        append_tree_rows(a.k_new, a.v_new, a.k_cache_w, a.v_cache_w, a.block_table + (long long)b * a.max_blocks, b, L,
                         N, a.Hkv * a.D * 2, a.bs_log2, ((long long)a.num_blocks << a.bs_log2) * a.Hkv * a.D * 2 / 16,
                         (long long)a.B * N * a.Hkv * a.D * 2 / 16, a.seq_err + b);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, int nm_max) {
    constexpr int HALVES = D / 64;
    constexpr uint32_t SLOT = 128u * D * 2u;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const TcLayout lay = tc_layout<D>(nm_max);
    const int nslots = lay.slots;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    int8_t* s_par = reinterpret_cast<int8_t*>(smem + lay.misc + kMiscPar);  // [2][128]
    volatile int* s_meta = reinterpret_cast<volatile int*>(smem + lay.misc + kMiscMeta);  // [kMaxSlots]
    int* s_sched = reinterpret_cast<int*>(smem + lay.misc + kMiscSched);
    int* s_blk0 = reinterpret_cast<int*>(smem + lay.misc + kMiscBlk0);  // [16]
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + lay.bars + 8 * Bars::kCount);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + lay.bars + 8 * Bars::kCount + 4);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [=](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrg = a.n_rgroups;
    const int rg = blockIdx.x % nrg, lane_c = blockIdx.x / nrg;
    const int N = a.N;
    const int bs = 1 << a.bs_log2;
    const int r_base = rg * 256;
    const int nm = min(2, (a.R - r_base + 127) / 128);

    // ---- set-up: barriers, TMEM, where this CTA's tiles start
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
        mbar_init(bar(Bars::kQ), 128 * nm);
        mbar_init(bar(Bars::kDone), 1);
        mbar_init(bar(Bars::kStall), 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), 512);
        tmem_relinquish();
    }
    pdl_launch_dependents();  // the check kernel before it has started: the schedule needs nothing from it
    if (warp == 2) find_start(a, lane_c, s_sched, s_blk0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int count = s_sched[5];  // tiles of this CTA
    const TileIt it0{s_sched[0], s_sched[1], s_sched[2], s_sched[3], s_sched[4]};
    int my_err = 0;
    int err_b = it0.b;  // sequence flagged if a wait of this thread gives up

    if (warp < 4) regs_dec<kRegsProducer>();  // warpgroup 0: producer, MMA issuer, two idle warps
    if (warp == 0) {
        // ============================ TMA producer (whole warp: lane j loads the id of
        // the tile's j-th cache block and issues that block's boxes).  The next tile's
        // block ids are loaded while the current tile's fills wait for their slots.
        TileIt it = it0;
        int blk = (count > 0 && lane < 16) ? s_blk0[lane] : 0;  // looked up during set-up
        const uint64_t kv_policy = l2_evict_first_policy();  // every K/V row is read once
        int seg = 0;
        bool appended = a.k_new == nullptr;  // the tree rows this kernel reads are in the cache
        int issued = 0;                      // fills issued so far
        for (int jt = 0; jt < count && !my_err; ++jt) {
            if (jt > 0 && it.t == 0) ++seg;
            const bool first = (jt == 0) || (it.t == 0);
            const int t0 = it.t * kTileKeys;
            if (!appended && t0 + kTileKeys > it.L) {
                // a tile with tree keys: the check kernel before this one in the stream has
                // written them (its memory is visible once it has completed); the copies
                // then read them through the async proxy
                pdl_wait();
                asm volatile("fence.proxy.async.global;" ::: "memory");
                appended = true;
            }
            const int nblk = (min(t0 + kTileKeys, it.L + N) - t0 + bs - 1) >> a.bs_log2;
            const int g = it.g;
            const int blk_cur = blk;
            err_b = it.b;
            if (jt + 1 < count) {
                it.next(a);
                const int u0 = it.t * kTileKeys;
                const int nb = (min(u0 + kTileKeys, it.L + N) - u0 + bs - 1) >> a.bs_log2;
                blk = lane < nb ? __ldg(a.block_table + (long long)it.b * a.max_blocks + (u0 >> a.bs_log2) + lane) : 0;
            }
#pragma unroll 1
            for (int kv = 0; kv < 2; ++kv) {
                const int f = 2 * jt + kv;
                const int slot = f % nslots, use = f / nslots;
                if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(Bars::kEmpty + slot), (use - 1) & 1, s_abort))) {
                    my_err = 1;
                    break;
                }
                const CUtensorMap* map = kv ? &tmv : &tmk;
                const uint32_t dst = smem_u32(smem + lay.ring + slot * SLOT);
                if (lane == 0) {
                    if (kv == 0) s_meta[slot] = (seg << 1) | (first ? 1 : 0);  // read by the MMA issuer
                    mbar_expect_tx(bar(Bars::kFull + slot), static_cast<uint32_t>(nblk * bs * 128 * HALVES));
                }
                __syncwarp();
                if (lane < nblk) {  // a 128-key tile spans at most 128 / 8 = 16 blocks
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh)
                        tma_load_3d(dst + hh * kHalfBytes + lane * bs * 128, map, bar(Bars::kFull + slot), hh * 64, g,
                                    blk_cur * bs, kv_policy);
                }
                issued = f + 1;
            }
            if (jt == 0 && count > 1 && count <= kFirstTileAloneMaxTiles && !my_err &&
                !__all_sync(0xffffffffu, mbar_wait(bar(Bars::kFull + 0), 0, s_abort)))
                my_err = 1;
        }
        // never leave with copies in flight: wait for the latest issued fill of every slot
        // (after an abort, fills that were never issued are not waited for)
        if (lane == 0) {
            for (int f = max(0, issued - nslots); f < issued; ++f) {
                volatile int never = 0;
                if (!mbar_wait(bar(Bars::kFull + f % nslots), (f / nslots) & 1, &never)) my_err = 1;
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer
        if (lane == 0 && count > 0) {
            constexpr uint32_t idS = idesc_bf16(128, 128, false);
            constexpr uint32_t idO = idesc_bf16(128, D, true);
            const uint32_t q_base = smem_u32(smem + lay.q0);
            const uint32_t ring_base = smem_u32(smem + lay.ring);
            // The descriptors are built once: a descriptor's start-address field is the
            // byte address >> 4 in its low bits, so the descriptor of (base + off) is the
            // base descriptor + off / 16 (every offset here is a multiple of 16 and all
            // addresses stay below 2^18).  Each MMA then costs one 64-bit add per operand.
            const uint64_t dQ = sdesc_sw128(q_base, 16, 1024);       // K-major Q tiles
            const uint64_t dK = sdesc_sw128(ring_base, 16, 1024);    // K-major K tiles
            const uint64_t dV = sdesc_sw128(ring_base, kHalfBytes, 1024);  // MN-major V tiles
            // S buffer sb (TMEM columns sb*128) = Q tile qm . K^T
            auto issue_S = [=](int qm, int sb, int slot) {
                const uint64_t qa = dQ + ((qm * (128u * D * 2u)) >> 4);
                const uint64_t kb = dK + ((slot * SLOT) >> 4);
                const uint32_t d = tmem + sb * 128;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off16 = ((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4;
                    mma_bf16(d, qa + off16, kb + off16, idS, k > 0);
                }
            };
            // O tile om += P . V, P in TMEM over S buffer pb's columns (16 keys = 8 columns per MMA)
            auto issue_PV = [=](int om, int pb, int slot, bool acc_first) {
                const uint64_t vb = dV + ((slot * SLOT) >> 4);
                const uint32_t d = tmem + 256 + om * D, pa = tmem + pb * 128;
#pragma unroll
                for (int k = 0; k < kTileKeys / 16; ++k)
                    mma_bf16_ts(d, pa + k * 8, vb + ((k * 16 * 128) >> 4), idO, (acc_first || k > 0) ? 1u : 0u);
            };
            // K tile of CTA tile jt in its slot; a tile that starts a segment also waits
            // for that segment's Q.  *first = the tile starts a segment.
            int q_seg = -1;
            auto wait_K = [&](int jt, bool* first) -> bool {
                const int f = 2 * jt;
                if (!mbar_wait(bar(Bars::kFull + f % nslots), (f / nslots) & 1, s_abort)) return false;
                const int meta = s_meta[f % nslots];
                *first = (meta & 1) != 0;
                const int sg = meta >> 1;
                if (sg != q_seg) {
                    if (!mbar_wait(bar(Bars::kQ), sg & 1, s_abort)) return false;
                    q_seg = sg;
                }
                tc_fence_after();
                return true;
            };
            bool ok = true;
            if (nm == 2) {
                // two M tiles ping-pong: one tile's softmax overlaps the other's MMAs
                bool fcur = false;
                ok = wait_K(0, &fcur);
                if (ok) {
                    for (int m = 0; m < nm; ++m) {
                        issue_S(m, m, 0);
                        mma_commit(bar(Bars::kS + m));
                    }
                    mma_commit(bar(Bars::kEmpty + 0));
                }
                for (int jt = 0; jt < count && ok; ++jt) {
                    const int fV = 2 * jt + 1, fK = 2 * jt + 2;
                    const int sV = fV % nslots, sK = fK % nslots;
                    const bool nxt = jt + 1 < count;
                    // everything this tile's products read besides P is waited for first, so each
                    // M tile's PV and next S go to the tensor pipe back to back
                    ok = mbar_wait(bar(Bars::kFull + sV), (fV / nslots) & 1, s_abort);
                    bool fnext = false;
                    if (ok && nxt) ok = wait_K(jt + 1, &fnext);
                    tc_fence_after();
                    for (int m = 0; m < nm && ok; ++m) {
                        ok = mbar_wait(bar(Bars::kP + m), jt & 1, s_abort);
                        if (!ok) break;
                        tc_fence_after();
                        issue_PV(m, m, sV, !fcur);
                        if (nxt) issue_S(m, m, sK);
                        mma_commit(bar(Bars::kO + m));
                        if (nxt) mma_commit(bar(Bars::kS + m));
                        if (m == nm - 1) mma_commit(bar(Bars::kEmpty + sV));  // V_jt's last reader issued
                    }
                    if (!ok) break;
                    if (jt + 1 < count) mma_commit(bar(Bars::kEmpty + fK % nslots));
                    fcur = fnext;
                }
            } else {
                // one M tile: S is double-buffered across key tiles (tile jt in buffer jt & 1),
                // so S(jt+1) is computed while tile jt's softmax runs.  K fills are consumed
                // ahead of V fills (K0, K1, V0, K2, V1, ...); the ring holds >= 3 slots.
                bool f0 = false, f1 = false;  // the tile in S buffer 0 / 1 starts a segment
                for (int jj = 0; jj < 2 && jj < count && ok; ++jj) {
                    bool fl = false;
                    ok = wait_K(jj, &fl);
                    if (!ok) break;
                    issue_S(0, jj, (2 * jj) % nslots);
                    mma_commit(bar(Bars::kS + jj));
                    mma_commit(bar(Bars::kEmpty + (2 * jj) % nslots));
                    if (jj) f1 = fl;
                    else f0 = fl;
                }
                for (int jt = 0; jt < count && ok; ++jt) {
                    const int b2 = jt & 1;
                    const int fV = 2 * jt + 1, fK = 2 * jt + 4;
                    ok = mbar_wait(bar(Bars::kFull + fV % nslots), (fV / nslots) & 1, s_abort) &&
                         mbar_wait(bar(Bars::kP + b2), (jt >> 1) & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_PV(0, b2, fV % nslots, !(b2 ? f1 : f0));
                    mma_commit(bar(Bars::kO + 0));
                    mma_commit(bar(Bars::kEmpty + fV % nslots));
                    if (jt + 2 < count) {
                        bool fl = false;
                        ok = wait_K(jt + 2, &fl);
                        if (!ok) break;
                        issue_S(0, b2, fK % nslots);  // after PV(jt) has read P(jt) from this buffer
                        mma_commit(bar(Bars::kS + b2));
                        mma_commit(bar(Bars::kEmpty + fK % nslots));
                        if (b2) f1 = fl;
                        else f0 = fl;
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
        regs_inc<kRegsSoftmax>();  // both softmax warpgroups, also the second one when it has no M tile
        if ((warp - 4) / 4 < nm) {
        // ============================ softmax warpgroups (warpgroup wg < nm)
        const int wg = (warp - 4) >> 2;
        const int nthr = 128 * nm;           // softmax threads taking part
        const int stid = tid - 128;          // 0 .. nthr-1
        const int tw = stid - wg * 128;      // TMEM lane = tile row handled by this thread
        // A partial M tile deals its rows round-robin over the four 32-lane quadrants of
        // TMEM (tile row tw holds row 4*(tw%32) + tw/32), so all four softmax warps share
        // the work; a full tile keeps the identity order.
        const int rows_here = min(128, a.R - r_base - wg * 128);
        const int rl = rows_here < 128 ? 4 * (tw & 31) + (tw >> 5) : tw;
        const int r = r_base + wg * 128 + rl;
        const bool valid = rl < rows_here;
        const int n = valid ? r / a.G : 0;
        const int hj = valid ? r % a.G : 0;  // head within the GQA group
        const bool warp_active = __any_sync(0xffffffffu, valid);
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS0 = tmem + lane_base;
        const uint32_t tO = tmem + lane_base + 256 + wg * D;
        const float sl2 = a.scale_log2;
        const long long s_first = reinterpret_cast<const long long*>(s_sched)[3];  // global index of tile 0
        const long long T_all = reinterpret_cast<const long long*>(s_sched)[4];
        bool ok = true;

        // Q rows of unit (bq, gq) -> this warpgroup's shared tile, stored as 64-element
        // halves of [128 rows x 128 B] with the 128B swizzle (16-byte chunk c of row r at
        // chunk c ^ (r & 7)); the copies are issued by issue_q and become visible to the
        // MMA issuer with finish_q
        auto issue_q = [&](int bq, int gq) {
            // the row's swizzle phase goes through an opaque move, so the chunk addresses
            // are formed here instead of being kept in registers across the tile loop
            const uint32_t r7 = opaque_u32(static_cast<uint32_t>(tw & 7));
            const uint32_t dst = smem_u32(smem + lay.q0 + wg * (128u * D * 2u)) + (tw >> 3) * 1024u + r7 * 128u;
            const long long qrow = (((long long)bq * N + n) * a.Hq + gq * a.G + hj) * D;
            const bool take = valid && TSV_IN_BOUNDS(qrow + D - 1, (long long)a.B * N * a.Hq * D, a.seq_err + bq);
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + (take ? qrow : 0));
#pragma unroll
            for (int qq = 0; qq < D / 8; ++qq)
                cp_async16(dst + (qq >> 3) * kHalfBytes + (((qq & 7) ^ r7) << 4), src + qq, take);
        };
        auto finish_q = [&]() {
            cp_async_wait_all();
            fence_proxy_async_smem();
            mbar_arrive(bar(Bars::kQ));
        };

        TileIt it = it0;
        int jt = 0, seg = 0;
        // parent of node stid in the coming segment's sequence (loaded one segment ahead)
        int par_next = 0;
        if (count > 0) {
            issue_q(it.b, it.g);
            if (stid < N) par_next = __ldg(a.parent + (long long)it.b * N + stid);
            finish_q();
        }
        while (jt < count) {
            // ---- segment: tiles [t_first, t_first + ntl) of unit (b, g)
            const int b = it.b, g = it.g, L = it.L, Tb = it.Tb, t_first = it.t;
            const int ntl = min(Tb - t_first, count - jt);
            const bool whole = (t_first == 0) && (ntl == Tb);
            const long long unit_first = s_first + jt - t_first;  // global index of the unit's tile 0
            const int par_cur = par_next;
            // the Q rows and parents of the next segment's unit are fetched during this
            // segment's last tile, once that tile's S product (the last reader of Q) is done
            const bool more = jt + ntl < count;
            err_b = b;
            if (t_first == 0 && stid == 0 &&
                TSV_IN_BOUNDS(((long long)b * a.Hkv + g) * nrg + rg, (long long)a.B * a.Hkv * nrg, a.seq_err + b)) {
                // this lane holds the unit's first piece: record where its pieces are
                int* ui = a.unit_info + (((long long)b * a.Hkv + g) * nrg + rg) * kUnitInfoInts;
                ui[0] = lane_c;
                ui[1] = lane_of_tile(unit_first + Tb - 1, T_all, a.lanes);
                ui[2] = seg == 0 ? 0 : 1;
                ui[3] = 0;
                reinterpret_cast<long long*>(ui)[2] = T_all;
            }
            // ancestor mask of this row's node (tree keys only)
            uint32_t anc0 = 0u, anc1 = 0u, anc2 = 0u, anc3 = 0u;
            if ((long long)(t_first + ntl) * kTileKeys > L) {
                int8_t* par = s_par + (seg & 1) * 128;
                if (stid < N) par[stid] = static_cast<int8_t>(par_cur);  // N <= 128 <= softmax threads
                named_bar_sync(1, nthr);
                if (valid) {
                    int x = n;
                    for (int step = 0; step <= N && x >= 0 && x < N; ++step) {
                        const uint32_t bit = 1u << (x & 31);
                        const int w = x >> 5;
                        anc0 |= w == 0 ? bit : 0u;
                        anc1 |= w == 1 ? bit : 0u;
                        anc2 |= w == 2 ? bit : 0u;
                        anc3 |= w == 3 ? bit : 0u;
                        x = par[x];
                    }
                }
            }
            float m_run = -INFINITY, l_run = 0.0f;
            for (int i = 0; i < ntl; ++i, ++jt) {
                if (!ok) continue;
                const int t0 = (t_first + i) * kTileKeys;
                // S/P buffer of this tile: the warpgroup's own with two M tiles; alternating
                // buffers (double-buffered S) with one
                const int sb = nm == 2 ? wg : (jt & 1);
                const uint32_t sphase = nm == 2 ? (jt & 1) : ((jt >> 1) & 1);
                const uint32_t tS = tS0 + sb * 128;
#ifdef TSV_TEST_HOOKS
                // the stalled wait: warpgroup 0's first S never arrives, the wait gives up
                const bool stall = g_test_stall != 0 && jt == 0 && wg == 0;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(stall ? Bars::kStall : Bars::kS + sb), sphase, s_abort));
#else
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bars::kS + sb), sphase, s_abort));
#endif
                if (!ok) {
                    *s_abort = 1;
                    continue;
                }
                tc_fence_after();
                const bool last_of_seg = (i == ntl - 1);
                if (last_of_seg && more) {
                    TileIt nx = it;
                    nx.next_unit(a);
                    issue_q(nx.b, nx.g);
                    if (stid < N) par_next = __ldg(a.parent + (long long)nx.b * N + stid);
                }
                if (warp_active) {
                    // One pass over the S row: all 128 scores come out of TMEM under one wait
                    // and stay in registers; keys off the row's path (a tile that reaches past
                    // the prefix) become -inf there; the raw max by three-input maxima; then
                    // P = 2^(s*scale - m) with the scale and offset applied to pairs of
                    // scores at a time, summed in pairs, packed to bf16 pairs over the first
                    // 64 columns.
                    uint32_t sv[128];
                    tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[64]));
                    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sv[96]));
                    tmem_wait_ld();
                    if (t0 + kTileKeys > L) {
#pragma unroll
                        for (int w4 = 0; w4 < 4; ++w4) {
                            const uint32_t vw = vis_word(t0 + 32 * w4 - L, anc0, anc1, anc2, anc3);
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc)
                                sv[32 * w4 + cc] = ((vw >> cc) & 1u) ? sv[32 * w4 + cc] : 0xff800000u;  // -inf
                        }
                    }
                    float mxa[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) mxa[q] = -INFINITY;
                    if (valid) {
#pragma unroll
                        for (int cc = 0; cc < 128; cc += 16)
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                mxa[q] = max3f(mxa[q], __uint_as_float(sv[cc + 2 * q]), __uint_as_float(sv[cc + 2 * q + 1]));
                    }
                    const float mx_raw = max3f(max3f(mxa[0], mxa[1], mxa[2]), max3f(mxa[3], mxa[4], mxa[5]),
                                               fmaxf(mxa[6], mxa[7]));
                    const float mx = mx_raw * sl2;  // scale > 0: max commutes with it
                    // within a segment, the PV product of the previous tile must be done
                    // before O is rescaled (a segment's first PV overwrites O).  With two M
                    // tiles that is implied by the S just waited for: its issuer committed it
                    // after that PV (a commit covers every earlier product of the issuing
                    // thread).  With one, S is double-buffered and was issued before that PV.
                    if (i > 0 && nm == 1) {
                        ok = __all_sync(0xffffffffu, mbar_wait(bar(Bars::kO + wg), (jt - 1) & 1, s_abort));
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
                    const unsigned long long sc2 = f2_pack(sl2, sl2), off2 = f2_pack(-m_run, -m_run);
                    unsigned long long la2[4] = {0ull, 0ull, 0ull, 0ull};  // (0.0f, 0.0f) pairs
                    uint32_t w[64];
#pragma unroll
                    for (int q = 0; q < 64; ++q) {
                        // a hidden key's -inf score gives 2^-inf = 0
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * q]), __uint_as_float(sv[2 * q + 1])), sc2, off2),
                                  x0, x1);
                        const float p0 = live ? ex2(x0) : 0.0f;
                        const float p1 = live ? ex2(x1) : 0.0f;
                        la2[q & 3] = f2_add(la2[q & 3], f2_pack(p0, p1));
                        __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
                        w[q] = *reinterpret_cast<uint32_t*>(&pk);
                    }
                    tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&w[0]));
                    tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&w[32]));
                    tmem_wait_st();
                    float s0, s1, s2, s3, s4, s5, s6, s7;
                    f2_unpack(la2[0], s0, s1);
                    f2_unpack(la2[1], s2, s3);
                    f2_unpack(la2[2], s4, s5);
                    f2_unpack(la2[3], s6, s7);
                    l_run += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
                }
                // a unit's last tile: V rows past the key range are zeroed before the PV
                // product (they may hold stale or foreign data; P is 0 there but 0 * NaN is NaN)
                if (wg == 0 && L + N - t0 < kTileKeys) {
                    const int fV = 2 * jt + 1;
                    ok = ok && mbar_wait(bar(Bars::kFull + fV % nslots), (fV / nslots) & 1, s_abort);
                    if (ok) {
                        // rows [L + N - t0, 128) of both halves; a row is HALVES * 8 chunks of 16 B
                        constexpr int kRowChunks = HALVES * 8, kRowsPerStep = 128 / kRowChunks;
                        uint8_t* vt = smem + lay.ring + (fV % nslots) * SLOT + ((tw % kRowChunks) >> 3) * kHalfBytes +
                                      (tw & 7) * 16;
                        for (int row = L + N - t0 + tw / kRowChunks; row < kTileKeys; row += kRowsPerStep)
                            *reinterpret_cast<uint4*>(vt + row * 128) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();  // the zeroed V rows, written through the generic proxy
                tc_fence_before();
                mbar_arrive(bar(Bars::kP + sb));
                if (!ok) *s_abort = 1;
                if (last_of_seg && more) finish_q();  // the next segment's Q rows are in place
            }
            // ---- epilogue: O / l of this segment
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bars::kO + wg), (jt - 1) & 1, s_abort));
                tc_fence_after();
                if (!ok) *s_abort = 1;
            }
            const int side = seg == 0 ? 0 : 1;  // a piece is this CTA's first or its last segment
            if (ok && warp_active) {
                const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;  // a piece may see no key of a row
                const long long orow = (((long long)b * N + n) * a.Hq + g * a.G + hj) * D;
                const long long prow = ((long long)blockIdx.x * 2 + side) * a.rows_item + wg * 128 + rl;
                const bool in_bounds =
                    !valid || (whole ? TSV_IN_BOUNDS(orow + D - 1, (long long)a.B * N * a.Hq * D, a.seq_err + b)
                                     : TSV_IN_BOUNDS(prow, 2LL * gridDim.x * a.rows_item, a.seq_err + b));
#pragma unroll 1
                for (int q4 = 0; q4 < D / 32; ++q4) {
                    uint32_t ov[32];
                    tmem_ld32(tO + q4 * 32, ov);
                    tmem_wait_ld();
                    if (valid && in_bounds) {
                        if (whole) {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + q4 * 32);
#pragma unroll
                            for (int v8 = 0; v8 < 4; ++v8) {
                                uint32_t w[4];
#pragma unroll
                                for (int e2 = 0; e2 < 4; ++e2) {
                                    __nv_bfloat162 pk =
                                        __floats2bfloat162_rn(__uint_as_float(ov[v8 * 8 + 2 * e2]) * inv,
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
                if (valid && !whole && in_bounds) {
                    a.part_m[prow] = m_run;
                    a.part_l[prow] = l_run;
                }
            }
            if (more) it.next_unit(a);
            ++seg;
        }
        if (!ok) my_err = 1;
        }
    }
    // the check kernel has written seq_err before this CTA completes (and so before the
    // merge kernel runs, or a timeout flag is added to it)
    pdl_wait();
    if (my_err) {
        *s_abort = 1;
        atomicOr(&a.seq_err[err_b], TSV_DERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Merge of the units that straddle lanes (log-sum-exp over their pieces).  One CTA per
// (unit, block of 32 rows); 8 threads per row, each owning D / 8 consecutive columns,
// so a row's 8 threads read its partial rows as one coalesced run.  Runs after the
// attention kernel (programmatic dependent launch: it waits for that kernel's writes).
template <int D>
__global__ void __launch_bounds__(256) attn_tc_merge_kernel(const AttnArgs a) {
    constexpr int C = D / 8;  // columns per thread
    pdl_wait();
    pdl_launch_dependents();
    const int nrg = a.n_rgroups;
    const int u = blockIdx.x;
    const int rg = u % nrg, g = (u / nrg) % a.Hkv, b = u / (nrg * a.Hkv);
    const int* ui = a.unit_info + (long long)u * kUnitInfoInts;
    const int e = a.seq_err[b];
    const int c_first = ui[0], c_last = ui[1], sd0 = ui[2];
    const long long T_all = reinterpret_cast<const long long*>(ui)[2];
    if (e & ~TSV_DERR_TIMEOUT) {  // flagged by the check kernel: this block's rows become NaN
        const int r_base = rg * 256, rows_rg = min(256, a.R - r_base);
        const int rr = blockIdx.y * 32 + (threadIdx.x >> 3), c0 = (threadIdx.x & 7) * C;
        if (rr < rows_rg) {
            const int r = r_base + rr;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                                 (((long long)b * a.N + r / a.G) * a.Hq + g * a.G + r % a.G) * D + c0;
            const __nv_bfloat16 nan = __float2bfloat16_rn(__int_as_float(0x7fc00000));
#pragma unroll
            for (int q = 0; q < C; ++q) dst[q] = nan;
        }
        return;
    }
    if (e != 0) return;  // timed out: outputs are not valid
    if (c_last <= c_first || c_first < 0 || c_last >= a.lanes || T_all < 1) return;  // one piece: written directly
    const int r_base = rg * 256;
    const int rows_rg = min(256, a.R - r_base);
    const int rr = blockIdx.y * 32 + (threadIdx.x >> 3), c0 = (threadIdx.x & 7) * C;
    if (rr >= rows_rg) return;
    const bool dense = T_all >= a.lanes;  // every lane has a non-empty run
    float acc[C];
#pragma unroll
    for (int q = 0; q < C; ++q) acc[q] = 0.0f;
    float M = -INFINITY, W = 0.0f;
    if (dense && c_last - c_first < 4) {
        // up to four pieces: every load is issued before any is used
        constexpr int P = 4;
        float lk[P], mk[P];
        float4 o[P][C / 4];
#pragma unroll
        for (int k = 0; k < P; ++k) {
            lk[k] = 0.0f;
            mk[k] = -INFINITY;
            if (c_first + k <= c_last &&
                TSV_IN_BOUNDS(((long long)((c_first + k) * nrg + rg) * 2 + (k == 0 ? sd0 : 0)) * a.rows_item + rr,
                              2LL * a.lanes * nrg * a.rows_item, a.seq_err + b)) {
                const long long pr = ((long long)((c_first + k) * nrg + rg) * 2 + (k == 0 ? sd0 : 0)) * a.rows_item + rr;
                lk[k] = __ldg(a.part_l + pr);
                mk[k] = __ldg(a.part_m + pr);
                const float4* src = reinterpret_cast<const float4*>(a.part_o + pr * D + c0);
#pragma unroll
                for (int q = 0; q < C / 4; ++q) o[k][q] = __ldg(src + q);
            }
        }
#pragma unroll
        for (int k = 0; k < P; ++k)
            if (lk[k] > 0.0f) M = fmaxf(M, mk[k]);
#pragma unroll
        for (int k = 0; k < P; ++k) {
            const float wk = lk[k] > 0.0f ? lk[k] * exp2f(mk[k] - M) : 0.0f;  // a piece may see no key of a row
            W += wk;
            if (wk > 0.0f) {
#pragma unroll
                for (int q = 0; q < C / 4; ++q) {
                    acc[4 * q] = fmaf(wk, o[k][q].x, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(wk, o[k][q].y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(wk, o[k][q].z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(wk, o[k][q].w, acc[4 * q + 3]);
                }
            }
        }
    } else {
        for (int k = c_first; k <= c_last; ++k) {
            if (!dense && lane_start(k + 1, T_all, a.lanes) == lane_start(k, T_all, a.lanes)) continue;
            const long long pr = ((long long)(k * nrg + rg) * 2 + (k == c_first ? sd0 : 0)) * a.rows_item + rr;
            const float lk = __ldg(a.part_l + pr), mk = __ldg(a.part_m + pr);
            if (!(lk > 0.0f)) continue;
            if (mk > M) {
                W = W * exp2f(M - mk) + lk;
                M = mk;
            } else {
                W += lk * exp2f(mk - M);
            }
        }
        for (int k = c_first; k <= c_last; ++k) {
            if (!dense && lane_start(k + 1, T_all, a.lanes) == lane_start(k, T_all, a.lanes)) continue;
            const long long pr = ((long long)(k * nrg + rg) * 2 + (k == c_first ? sd0 : 0)) * a.rows_item + rr;
            const float lk = __ldg(a.part_l + pr);
            if (!(lk > 0.0f)) continue;
            const float wk = lk * exp2f(__ldg(a.part_m + pr) - M);
            const float4* src = reinterpret_cast<const float4*>(a.part_o + pr * D + c0);
#pragma unroll
            for (int q = 0; q < C / 4; ++q) {
                const float4 o = __ldg(src + q);
                acc[4 * q] = fmaf(wk, o.x, acc[4 * q]);
                acc[4 * q + 1] = fmaf(wk, o.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(wk, o.z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(wk, o.w, acc[4 * q + 3]);
            }
        }
    }
    const float winv = 1.0f / W;
    const int r = r_base + rr;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                          (((long long)b * a.N + r / a.G) * a.Hq + g * a.G + r % a.G) * D + c0);
#pragma unroll
    for (int q = 0; q < C / 8; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 pk = __floats2bfloat162_rn(acc[8 * q + 2 * e] * winv, acc[8 * q + 2 * e + 1] * winv);
            w[e] = *reinterpret_cast<uint32_t*>(&pk);
        }
        dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
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

// The tensor maps of the most recent caches this host thread used (encoding them costs
// microseconds of host time per call).
struct MapCache {
    const void* k = nullptr;
    const void* v = nullptr;
    int D = 0, Hkv = 0, bs = 0;
    long long rows = 0;
    CUtensorMap mk, mv;
};

template <int D>
cudaError_t launch_tc_inst(const AttnArgs& a, cudaStream_t stream) {
    thread_local MapCache mc;
    const long long rows = static_cast<long long>(a.num_blocks) << a.bs_log2;
    const int bs = 1 << a.bs_log2;
    if (mc.k != a.k_cache || mc.v != a.v_cache || mc.D != D || mc.Hkv != a.Hkv || mc.bs != bs || mc.rows != rows) {
        mc.k = nullptr;
        if (!make_cache_map(&mc.mk, a.k_cache, D, a.Hkv, rows, bs) || !make_cache_map(&mc.mv, a.v_cache, D, a.Hkv, rows, bs))
            return cudaErrorInvalidValue;
        mc.k = a.k_cache;
        mc.v = a.v_cache;
        mc.D = D;
        mc.Hkv = a.Hkv;
        mc.bs = bs;
        mc.rows = rows;
    }
    const CUtensorMap& mk = mc.mk;
    const CUtensorMap& mv = mc.mv;
    cudaError_t e = launch_pdl(attn_tc_check_kernel, dim3(static_cast<unsigned>(a.B)), dim3(a.k_new ? 256 : 128), 0,
                               stream, 1u, a);
    if (e != cudaSuccess) return e;
    const int nm_max = a.R > 128 ? 2 : 1;
    const TcLayout lay = tc_layout<D>(nm_max);
    // the kernel's dynamic shared memory limit, raised once per device and host thread
    thread_local int smem_dev = -1, smem_set = -1;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != smem_dev || static_cast<int>(lay.total) > smem_set) {
        e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(lay.total));
        if (e != cudaSuccess) return e;
        smem_dev = dev;
        smem_set = static_cast<int>(lay.total);
    }
    e = launch_pdl(attn_tc_kernel<D>, dim3(static_cast<unsigned>(a.lanes * a.n_rgroups)), dim3(kThreads), lay.total,
                   stream, 1u, a, mk, mv, nm_max);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_tc_merge_kernel<D>,
                      dim3(static_cast<unsigned>(a.B * a.Hkv * a.n_rgroups), static_cast<unsigned>((a.rows_item + 31) / 32)),
                      dim3(256), 0, stream, 1u, a);
}

}  // namespace

bool attn_tc_supported(int D) { return D == 64 || D == 128; }

#ifdef TSV_TEST_HOOKS
// test build only: 1 = the next attention calls stall one wait until it times out
extern "C" int tsv_test_set_stall(int mode) {
    return (int)cudaMemcpyToSymbol(g_test_stall, &mode, sizeof(int));
}
#endif
int attn_tc_rows_per_cta() { return 256; }

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream) {
    return a.D == 64 ? launch_tc_inst<64>(a, stream) : launch_tc_inst<128>(a, stream);
}

}  // namespace tsv
