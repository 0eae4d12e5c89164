// moe_gemm_2sm.cu -- the grouped expert GEMMs for wide pair chunks (prefill
// and other batches with many pairs per expert) on CTA pairs, with the pairs
// on the MMA's M side: one tcgen05.mma.cta_group::2 multiplies 256 pair rows
// (128 in each CTA of the pair) by up to 256 weight rows (half of them in each
// CTA's shared memory), and every CTA's tensor memory receives its own 128
// pairs x all of the weight rows.
//
// Layer math ("Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Implementing multi-LoRA
// inference for MoE models in vLLM", Figure 1), per routed pair:
//   gate_up:  g = W1[e] x + B1[l][e] z1,  act = SiLU(g[0:I]) * g[I:2I]
//   down:     d = W2[e] act + B2[l][e] z2, pair_out = w * d
//
// Why this orientation.  On GB300 a ring stage of TMA copies costs about the
// same few hundred cycles whatever its size up to 64 KiB, so a wide-chunk
// GEMM is bound by its copies per MAC, not by the tensor pipe.  Here a task is
// (active expert, tile of weight rows, chunk of up to 256 pairs) and each K
// step issues two independent MMA chains of N = nu weight rows each: gate_up
// chain 0 the gate rows and chain 1 the up rows of nu intermediate units,
// down chain 0 and chain 1 two consecutive ranges of nu W2 rows.  Per K step
// a CTA copies its 128 pair rows and nu/2 rows of each chain (three boxes,
// at most 48 KiB) for 2 x 128 x nu x 64 MACs: twice the MACs per copied byte
// of a one-CTA tile of 128 weight rows.  Two independent chains keep the
// tensor pipe at its rate (one chain alone leaves gaps between dependent
// MMAs).  The two chains fill the 512 columns of tensor memory, so a task's
// epilogue does not overlap the next task's MMAs; it is short because each
// epilogue thread owns one pair and writes whole runs of its output row.
//
// gate_up puts a unit's gate value and its up value in the same thread (the
// same pair's TMEM lane, 256 columns apart), so SiLU(gate) * up is local.
//
// Experts whose pairs fill one 256-row chunk and part of a second (257 - 384
// pairs) may instead run in chunks of 256 + 128 pairs with chains of
// nu_t <= 160 rows: the last 128 pairs (64 per CTA) go through an M = 128
// MMA that reads the same weight stage, so the expert's weights stream once.
//
// LoRA, in the same orientation:
//   shrink items (the blog's shrink, section "Kernel optimizations"): the A
//     matrices of 256 / r consecutive (expert, adapter) buckets stacked on N
//     (r rows each, half of the buckets in each CTA) against the pair rows of
//     those buckets on M; each pair keeps the r columns of its own bucket.
//     Items are taken before every GEMM task; split over K when they are few
//     (the split that arrives last adds the partials in split order).
//   expand (the blog's fused LoRA add): extra K blocks of the base GEMM into
//     the same accumulators, A = zexp rows (each pair's z under its own
//     adapter's slot, zeros under the others) and B = the adapters' B rows of
//     the task's weight tile; a block holds 64 / r_pad consecutive adapters,
//     and only blocks with an adapter present in the chunk are issued.
//
// Roles in each CTA of the pair (one pair per two SMs, persistent; the
// leader's producer takes the next item from a device counter when it is
// ready for it, shrink items first, and hands its index to every role of
// both CTAs through a queue in each CTA's shared memory):
//   warp 0   TMA producer of this CTA's halves of every stage; the copies of
//            both CTAs count on the leader's (rank 0) full barrier, which the
//            leader arms with both byte counts;
//   warp 1   allocates the 512 TMEM columns (collectively with the peer); in
//            the leader one thread issues every MMA of the pair and commits
//            stage releases and accumulator completion to both CTAs;
//   warps 2-9 epilogue of this CTA's 128 TMEM lanes (= pairs); the peer's
//            warps free the accumulator on the leader's barrier;
//   warps 10-17 (FP8 weights only) expand the E4M3 codes the producer copies
//            into a stage's chain-row slots into bf16 weights, in place, and
//            tell the leader's MMA thread (wready).
// Every wait is bounded; on a timeout the CTA records kStatusTimeout, stops
// waiting, drains its copies, frees TMEM and exits at the final pair barrier.
#include "gemm_tasks.cuh"

namespace moelora {

namespace {

constexpr int kPairRows = 256;                  // pairs per chunk (M of one MMA over the pair)
constexpr int kTmem2 = 512;                     // the whole TMEM of the SM: one accumulator set
constexpr int kChain1Col = 256;                 // first TMEM column of chain 1
constexpr int kSlot = 128 * kBK * 2;            // 16 KiB: 128 rows of one 64-wide K step
constexpr int kStage2 = 3 * kSlot;              // pair rows, chain-0 rows, chain-1 rows
// Chunks of an expert in mode 1 hold up to 256 + 128 pairs: the last 128 (64
// per CTA) on an M = 128 MMA that reads the same weight stage.  Its tensor
// memory is 64 lanes x nu/2 columns per chain, so chains of nu_t <= 160 rows
// fit beside the main accumulators (2 nu_t + 2 nu_t / 2 <= 512).  The tail
// pair rows (and zexp rows) follow the main 128 in the stage; in mode 1 the
// chain rows start after them.
constexpr int kTailRows = 128;
constexpr int kChunkT = kPairRows + kTailRows;
constexpr int kXTail = kSlot;                   // tail pair rows in a stage (8 KiB)
constexpr int kC0T = kSlot + kSlot / 2;         // mode 1: chain-0 rows in a bf16 stage
// FP8 weights: a stage holds the pair rows (main and tail, 24 KiB) and the
// two chains' rows (16 KiB each, from kC0T); a base K step's codes are
// copied into the upper half of each chain's slot and expanded in place to
// bf16 by kConvWarps converter warps.
constexpr int kStageW8 = kC0T + 2 * kSlot;
constexpr int kCodeOff = kSlot / 2;            // a chain's codes inside its slot
constexpr int kConvWarps = 8;
constexpr int kConvWarp0 = 2 + kEpiWarps;      // first converter warp
constexpr int kThreadsW8 = (kConvWarp0 + kConvWarps) * 32;
constexpr int kMaxShrinkSlots = 32;             // buckets per shrink item: 256 / r with r >= 8
constexpr int kTaskQ2 = 8;                      // task queue slots (in each CTA of the pair)
// down epilogue: each warp turns its 32 pairs x 16 columns into whole
// 64-byte runs of 8 rows per store through a padded tile (row stride of 20
// floats: the 8 rows of a quarter-warp hit distinct banks)
constexpr int kTrStride = 20;
constexpr int kTrFloats = 32 * kTrStride;

template <bool B>
struct BoolC {
    static constexpr bool value = B;
};

// ---------------------------------------------------------------- CTA pair
__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same variable in the CTA of rank `rank`
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// wait with cluster-scope acquire: for phases completed by arrivals of the peer CTA
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kWaitRounds; i++) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 255u) == 0 && global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

// Tiled loads into this CTA's shared memory whose completion counts on an
// mbarrier of either CTA of the pair (`bar`: a shared::cluster address).
__device__ __forceinline__ void tma2_2d(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma2_3d(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma2_4d(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2,
                                        int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void tma2_5d(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2,
                                        int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

// TMEM of both CTAs, allocated and freed collectively (one warp in each CTA)
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T (M = 256 over the pair)
__device__ __forceinline__ void umma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on `bar` in both CTAs when every MMA issued so far has completed
__device__ __forceinline__ void umma2_commit_both(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane (warp-wide)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = __uint_as_float(r[i]);
}

// two fp32 -> two bf16 (round to nearest even) packed low, high: one cvt
// instruction (its first source goes to the upper half)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Task table (shared memory; every thread of the CTA builds it): per active
// expert its first pair row, pair count, chunk mode and the prefix sums of
// its tasks (weight tiles x chunks) and of its chunks.  Mode 0: chunks of 256
// pairs, chains of nu rows.  Mode 1: chunks of 256 + 128 pairs, chains of
// nu_t rows.  An expert takes mode 1 when it copies fewer rows that way: the
// stages of these GEMMs cost about their copied rows, and a copied weight
// row is shared by every pair of the chunk, so an expert with 257 - 384 pairs
// copies its weights once in mode 1 and twice in mode 0.
struct PairTable {
    unsigned long long* cmask;  // [chunks] adapters (< 64) with pairs in each (expert, chunk)
    int* e;     // [n_active]
    int* q0;    // [n_active]
    int* m;     // [n_active]
    int* md;    // [n_active] chunk mode
    int* cum;   // [n_active + 1] tasks before each expert
    int* ccum;  // [n_active + 1] chunks before each expert
};

struct PairTask {
    int e, mt, q0c, n_real, n_main, n_tail, chunk, split, mode, nu;
    __device__ void lookup(const PairTable& tt, int n_active, int ksplit, int nu0, int nu1, int t) {
        const int tile = t / ksplit;
        split = t % ksplit;
        int lo = 0, hi = n_active;  // last expert a with cum[a] <= tile
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tt.cum[mid] <= tile) lo = mid;
            else hi = mid;
        }
        mode = tt.md[lo];
        const int cap = mode ? kChunkT : kPairRows;
        const int m = tt.m[lo];
        const int nch = (m + cap - 1) / cap;
        const int loc = tile - tt.cum[lo];
        mt = loc / nch;
        const int ch = loc % nch;
        chunk = tt.ccum[lo] + ch;
        e = tt.e[lo];
        q0c = tt.q0[lo] + ch * cap;
        n_real = min(cap, m - ch * cap);
        n_main = min(n_real, kPairRows);
        n_tail = n_real - n_main;
        nu = mode ? nu1 : nu0;
    }
};

// nt0 / nt1: weight tiles of an expert in mode 0 / 1; nu1 = 0: mode 0 only
__device__ void build_pair_table(const TcArgs& a, const PairTable& tt, int n_active, int nt0, int nt1, int nu0,
                                 int nu1) {
    for (int ai = threadIdx.x; ai < n_active; ai += blockDim.x) {
        const int L1 = a.L + 1;
        const int e = a.active_experts[ai];
        const int q0 = a.compact_offset[e * L1];
        const int m = a.compact_offset[(e + 1) * L1] - q0;
        // rows a CTA copies per K step over all of the expert's tasks
        const int nch0 = (m + kPairRows - 1) / kPairRows;
        const long rows0 = (long)nch0 * nt0 * (128 + nu0);
        int mode = 0;
        if (nu1 > 0) {
            const int nch1 = (m + kChunkT - 1) / kChunkT;
            const int tails = m / kChunkT + (m % kChunkT > kPairRows ? 1 : 0);
            const long rows1 = (long)nt1 * ((long)nch1 * (128 + nu1) + (long)tails * (kTailRows / 2));
            mode = rows1 < rows0 ? 1 : 0;
        }
        const int nch = mode ? (m + kChunkT - 1) / kChunkT : nch0;
        tt.e[ai] = e;
        tt.q0[ai] = q0;
        tt.m[ai] = m;
        tt.md[ai] = mode;
        tt.cum[ai + 1] = (mode ? nt1 : nt0) * nch;
        tt.ccum[ai + 1] = nch;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < 2) {
        // warp 0 scans the task counts, warp 1 the chunk counts
        int* const arr = warp == 0 ? tt.cum : tt.ccum;
        int carry = 0;
        for (int base = 0; base < n_active; base += 32) {
            const int i = base + lane;
            int v = i < n_active ? arr[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, v, o);
                if (lane >= o) v += y;
            }
            if (i < n_active) arr[i + 1] = carry + v;
            carry += __shfl_sync(kFull, v, 31);
        }
        if (lane == 0) arr[0] = 0;
    }
    __syncthreads();
    if (a.chunk_masks) {
        // adapters with pairs in each (expert, chunk): one item per (expert,
        // adapter) bucket, OR-ed into the chunks the bucket's rows fall in
        const int n_chunks = tt.ccum[n_active];
        for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) tt.cmask[c] = 0ull;
        __syncthreads();
        for (int w = threadIdx.x; w < n_active * a.L; w += blockDim.x) {
            const int ai = w / a.L, l = w % a.L;
            const int b = tt.e[ai] * (a.L + 1) + l + 1;
            const int lo = a.compact_offset[b] - tt.q0[ai], hi = a.compact_offset[b + 1] - tt.q0[ai];
            const int cap = tt.md[ai] ? kChunkT : kPairRows;
            const int c0 = tt.ccum[ai];
            for (int ch = lo / cap; hi > lo && ch <= (hi - 1) / cap; ch++) atomicOr(&tt.cmask[c0 + ch], 1ull << l);
        }
        __syncthreads();
    }
}

// Shared memory after the stage ring: barriers, the TMEM base, shrink-slot
// tables and the task table.
struct Smem2 {
    uint8_t* ring;    // [NS][kStage2]; FP8 weights: [NS][kStageW8]
    uint64_t* full;   // [NS] leader: both CTAs' copies of stage s landed
    uint64_t* empty;  // [NS] the pair's MMAs are done with stage s
    uint64_t* wready; // FP8 weights: [NS] leader: both CTAs' converters are done with stage s
    uint64_t* cfull;  // FP8 weights: [NS] this CTA's codes of stage s landed (or the stage has none)
    uint64_t* tfull;  // accumulator ready for the epilogue
    uint64_t* tempty; // leader: accumulator drained by both CTAs' epilogues
    uint64_t* ebar;   // epilogue rendezvous
    uint64_t* cvbar;  // FP8 weights: converter rendezvous
    uint32_t* tmem_slot;
    uint64_t* tq_full;  // [kTaskQ2] task index of a queue slot written (in this CTA)
    uint64_t* tq_empty; // [kTaskQ2] leader: every consumer of both CTAs has read a slot
    int* tq;            // [kTaskQ2] task indices
    int* s_cb;        // [kMaxShrinkSlots] first row (relative to the item) of each slot's bucket
    int* s_ce;        // [kMaxShrinkSlots] one past its last row
    int* s_sl;        // [kMaxShrinkSlots] adapter of each slot
    int* s_misc;      // [4] shared verdicts
    float* tr;        // [kEpiWarps][kTrFloats] down epilogue transpose tiles
    PairTable tt;
};

__device__ inline Smem2 carve2(uint8_t* base, const TcArgs& a, int NS) {
    Smem2 m;
    m.ring = base;
    const int nw = a.w8 ? NS : 0;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + (size_t)NS * (a.w8 ? kStageW8 : kStage2));
    m.full = bars;
    m.empty = m.full + NS;
    m.wready = m.empty + NS;
    m.cfull = m.wready + nw;
    m.tfull = m.cfull + nw;
    m.tempty = m.tfull + 1;
    m.ebar = m.tempty + 1;
    m.cvbar = m.ebar + 1;
    m.tmem_slot = reinterpret_cast<uint32_t*>(m.cvbar + 1);
    m.tq_full = reinterpret_cast<uint64_t*>(m.tmem_slot + 4);
    m.tq_empty = m.tq_full + kTaskQ2;
    m.tq = reinterpret_cast<int*>(m.tq_empty + kTaskQ2);
    m.s_cb = m.tq + kTaskQ2;
    m.s_ce = m.s_cb + kMaxShrinkSlots;
    m.s_sl = m.s_ce + kMaxShrinkSlots;
    m.s_misc = m.s_sl + kMaxShrinkSlots;
    m.tt.cmask = reinterpret_cast<unsigned long long*>(m.s_misc + 4);
    m.tt.e = reinterpret_cast<int*>(m.tt.cmask + a.max_chunks);
    m.tt.q0 = m.tt.e + a.E;
    m.tt.m = m.tt.q0 + a.E;
    m.tt.md = m.tt.m + a.E;
    m.tt.cum = m.tt.md + a.E;
    m.tt.ccum = m.tt.cum + a.E + 1;
    m.tr = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(m.tt.ccum + a.E + 1) + 15) & ~uintptr_t(15));
    return m;
}

// Epilogue of shrink item t (accumulator used `use` times before), pairs on
// the lanes: this CTA's TMEM lane L holds item row rank * 128 + L, and r
// columns per slot s hold that row times the A matrix of slot s (slots
// 0 .. 128/r - 1 from column 0, the peer CTA's slots from column 128).
// A row keeps the columns of the slot whose bucket it belongs to (rows of
// base-only buckets between the item's buckets keep nothing).  Without a K
// split it writes z (fp32) and, for the tensor-core expand, zexp (bf16, the
// pair's own adapter slot); with one, its partial, and the split of this
// CTA's half that arrives last adds all partials in split order and writes
// z and zexp.  Each CTA then counts itself once in zdone.  False on a
// timeout (warp-uniform).
template <typename Rdv, typename Rel>
__device__ bool shrink_epilogue_m(const TcArgs& a, int t, int n_lora, int use, uint32_t tmem_base, int qd, int half,
                                  int lane, int etid, const Smem2& m, Rdv& rendezvous, Rel& release, int rank) {
    ShItem sh;
    sh.load(a, t, n_lora);
    const int r = a.r;
    // slot row ranges (after everyone is done with the previous item's)
    if (!rendezvous()) return false;
    if (etid < sh.nb) {
        const int bk = a.lora_buckets[sh.j0 + etid];
        m.s_cb[etid] = min(max(a.compact_offset[bk] - sh.q0c, 0), sh.n_real);
        m.s_ce[etid] = min(max(a.compact_offset[bk + 1] - sh.q0c, 0), sh.n_real);
        m.s_sl[etid] = bk % (a.L + 1) - 1;
    }
    if (!rendezvous()) return false;
    const int row = rank * 128 + qd * 32 + lane;      // row of the item held by this lane
    int my_s = -1;
    for (int s = 0; s < sh.nb; s++)
        if (row >= m.s_cb[s] && row < m.s_ce[s]) my_s = s;
    // the slots this warp's 32 rows touch (rows are in slot order)
    const int w_lo = rank * 128 + qd * 32, w_hi = w_lo + 31;
    int s_lo = sh.nb, s_hi = -1;
    for (int s = 0; s < sh.nb; s++) {
        if (m.s_ce[s] > w_lo && m.s_cb[s] <= w_hi) {
            s_lo = min(s_lo, s);
            s_hi = max(s_hi, s);
        }
    }
    const size_t q = (size_t)sh.q0c + row;
    float* dst = a.sh_ks > 1 ? a.zpart + (size_t)sh.sp * a.P * r : a.z;
    const int rp = expand_rpad(r);
    const bool zx = a.zexp != nullptr && a.sh_ks == 1;

    if (!__all_sync(kFull, mbar_wait(m.tfull, (uint32_t)use & 1u))) return false;
    tc_fence_after();
    const uint32_t t_lane = tmem_base + ((uint32_t)(qd * 32) << 16);
    // the two warps of a lane quadrant take alternate slots; slot s is column
    // range g * 128 + (s - g * g_cta) * r of the CTA g = s / g_cta that holds
    // its A rows (the N half of that CTA starts at column 128 g)
    const int g_cta = 128 / r;
    for (int s = s_lo + half; s <= s_hi; s += 2) {
        const int col = (s / g_cta) * 128 + (s % g_cta) * r;
        for (int j0 = 0; j0 < r; j0 += 8) {
            float v[8];
            tmem_ld8(t_lane + (uint32_t)(col + j0), v);
            if (my_s == s) {
                float4* zo = reinterpret_cast<float4*>(dst + q * r + j0);
                zo[0] = make_float4(v[0], v[1], v[2], v[3]);
                zo[1] = make_float4(v[4], v[5], v[6], v[7]);
                if (zx) {
                    uint4 pk;
                    pk.x = pack_bf16x2(v[0], v[1]);
                    pk.y = pack_bf16x2(v[2], v[3]);
                    pk.z = pack_bf16x2(v[4], v[5]);
                    pk.w = pack_bf16x2(v[6], v[7]);
                    *reinterpret_cast<uint4*>(a.zexp + ((size_t)m.s_sl[s] * a.P + q) * rp + j0) = pk;
                }
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release();
    __threadfence();
    if (!rendezvous()) return false;
    if (a.sh_ks > 1) {
        if (etid == 0) m.s_misc[1] = atomicAdd(&a.sh_counters[sh.i * 2 + rank], 1) == a.sh_ks - 1;
        if (!rendezvous()) return false;
        if (!m.s_misc[1]) return true;  // the last split of this CTA's half counts it
        __threadfence();
        // this CTA's rows, r / 4 float4 per row, summed in split order
        const int lo = min(rank * 128, sh.n_real), hi = min(rank * 128 + 128, sh.n_real);
        const int r4 = r / 4;
        const size_t split4 = (size_t)a.P * r / 4;
        const float4* src = reinterpret_cast<const float4*>(a.zpart);
        float4* zout = reinterpret_cast<float4*>(a.z);
        for (int i = etid; i < (hi - lo) * r4; i += kEpiWarps * 32) {
            const int rr = lo + i / r4, j4 = i % r4;
            const size_t at = ((size_t)sh.q0c + rr) * r4 + j4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sp = 0; sp < a.sh_ks; sp++) {
                const float4 v = __ldcg(src + sp * split4 + at);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            zout[at] = acc;
            if (a.zexp != nullptr) {
                int l = -1;
                for (int s = 0; s < sh.nb; s++)
                    if (rr >= m.s_cb[s] && rr < m.s_ce[s]) l = m.s_sl[s];
                if (l >= 0) {
                    uint2 pk;
                    pk.x = pack_bf16x2(acc.x, acc.y);
                    pk.y = pack_bf16x2(acc.z, acc.w);
                    *reinterpret_cast<uint2*>(a.zexp + ((size_t)l * a.P + sh.q0c + rr) * rp + j4 * 4) = pk;
                }
            }
        }
        __threadfence();
        if (!rendezvous()) return false;
    }
    if (etid == 0) atomicAdd(a.zdone, 1);
    return true;
}

// E4M3 codes -> bf16 of (scale * value): 16 codes (one 16-byte chunk of a
// staged row) into the two 16-byte chunks at `dst0` and `dst1`.
//
// A code b (sign bit, 4-bit exponent field f with bias 7, 3-bit mantissa m)
// placed in a bf16 as sign -> bit 15 and its other seven bits -> bits 10..4
// reads as a bf16 of exponent field f and mantissa m / 8: exactly
// value(b) * 2^-120, subnormal codes (f = 0) included, since both formats
// then scale m / 8 by their smallest exponent.  Two codes at a time: one
// byte permute puts them in the upper bytes of the two halves of a word, a
// shift and two logic ops move the bits, and one packed bf16 multiply by
// the row's factor gives the weights.  The factor is scale * 2^120 rounded
// once to bf16 (per row), so each weight is bf16(value * that), rounded
// once; when scale * 2^120 is beyond bf16's range the factor is
// scale * 2^64 and an exact second multiply by 2^56 follows.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// the two codes of w that `sel` picks, as bf16 bits of value * 2^-120 (low, high half)
__device__ __forceinline__ uint32_t e4m3x2_bits(uint32_t w, uint32_t sel) {
    const uint32_t t = __byte_perm(w, 0u, sel);
    return ((t >> 4) & 0x07F007F0u) | (t & 0x80008000u);
}

__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 c, uint32_t f_hi, uint32_t f_lo, bool two, uint4* dst0,
                                                uint4* dst1) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t lo = mul_bf16x2(e4m3x2_bits(w[i], 0x1404u), f_hi);  // codes 4i, 4i + 1
        uint32_t hi = mul_bf16x2(e4m3x2_bits(w[i], 0x3424u), f_hi);  // codes 4i + 2, 4i + 3
        if (two) {
            lo = mul_bf16x2(lo, f_lo);
            hi = mul_bf16x2(hi, f_lo);
        }
        o[2 * i] = lo;
        o[2 * i + 1] = hi;
    }
    *dst0 = make_uint4(o[0], o[1], o[2], o[3]);
    *dst1 = make_uint4(o[4], o[5], o[6], o[7]);
}

template <bool GATE_UP, bool W8>
__global__ void __launch_bounds__(W8 ? kThreadsW8 : kTcThreads, 1) k_moe_gemm_2sm(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int NS = a.nstages;
    Smem2 m = carve2(base, a, NS);
    const PairTable& tt = m.tt;
    const uint32_t rank = cta_rank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
            if (W8) {
                mbar_init(&m.wready[s], 2 * kConvWarps);  // the converter warps of both CTAs
                mbar_init(&m.cfull[s], 1);                 // this CTA's producer
            }
        }
        mbar_init(m.tfull, 1);
        mbar_init(m.tempty, 2 * kEpiWarps);
        mbar_init(m.ebar, kEpiWarps * 32);
        mbar_init(m.cvbar, kConvWarps * 32);
        // the task queue: one write per slot (the leader's producer, in both
        // CTAs); reads in each CTA by the MMA thread (leader) or the producer
        // (peer), every epilogue warp and, with FP8 weights, every converter warp
        for (int q = 0; q < kTaskQ2; q++) {
            mbar_init(&m.tq_full[q], 1);
            mbar_init(&m.tq_empty[q], 2 * (1 + kEpiWarps + (W8 ? kConvWarps : 0)));
        }
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc2(m.tmem_slot, kTmem2);
    if (warp == 0 && lane == 0) {
        if (!W8) prefetch_tensormap(&a.wmap);
        prefetch_tensormap(&a.xmap);
        if (a.nu_t) {
            if (!W8) prefetch_tensormap(&a.wmap_t);
            prefetch_tensormap(&a.xmap_t);
            if (a.tc_expand) {
                prefetch_tensormap(&a.bmap_t);
                prefetch_tensormap(&a.zxmap_t);
            }
            if (W8) prefetch_tensormap(&a.w8map_t);
        }
        if (a.sh_tasks) prefetch_tensormap(&a.amap);
        if (a.tc_expand) {
            prefetch_tensormap(&a.bmap);
            prefetch_tensormap(&a.zxmap);
        }
        if (W8) prefetch_tensormap(&a.w8map);
    }
    tc_fence_before();
    __syncthreads();
    // the peer's barriers exist before any arrival crosses the pair
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *m.tmem_slot;

    pdl_wait();
    pdl_trigger();

    // a task covers nu units (gate_up: the gate and the up rows of each) or
    // 2 * nu W2 rows (down), nu = a.nu for mode-0 chunks and a.nu_t for mode-1
    // chunks; each CTA copies nu / 2 rows of each chain
    const int nu0 = a.nu, nu1 = a.nu_t;
    const int N_out = GATE_UP ? a.I : a.H;
    const int K = GATE_UP ? a.H : a.I;
    const int tr0 = GATE_UP ? nu0 : 2 * nu0, tr1 = GATE_UP ? nu1 : 2 * nu1;
    const int nt0 = (N_out + tr0 - 1) / tr0;
    const int nt1 = nu1 > 0 ? (N_out + tr1 - 1) / tr1 : 0;
    const int nkb = (K + kBK - 1) / kBK;
    const int n_active = a.hdr->n_active;
    build_pair_table(a, tt, n_active, nt0, nt1, nu0, nu1);
    const int ksplit = a.ksplit;
    const bool shrink = a.sh_tasks != nullptr && a.r > 0;
    const bool expand = a.tc_expand != 0 && a.r > 0;
    const int sh_ks = a.sh_ks;
    const int n_sh_tasks = shrink ? a.hdr->n_shrink_tasks : 0;
    const int n_sh = n_sh_tasks * sh_ks;
    const int n_lora = shrink ? a.hdr->n_lora_buckets : 0;
    const int L1 = a.L + 1;
    const int g2 = a.r > 0 ? 128 / a.r : 0;  // shrink slots per CTA
    const int total = n_sh + tt.cum[n_active] * ksplit;
    const int t_first = (int)cluster_index(), t_step = (int)cluster_count();
    // Items are taken in order from a device counter by the leader's producer
    // when it is ready for the next one (so pairs that drew cheap items take
    // more), and handed to every role of both CTAs through the task queue;
    // without a counter they are dealt round-robin over the pairs.
    const bool dyn = a.task_counter != nullptr;
    const uint32_t lead_tq_empty = cluster_addr(m.tq_empty, 0);
    // the consumers' view of item `it`: one thread, or a whole warp (warp_call)
    auto take_task = [&](int it, bool& good, bool warp_call) -> int {
        good = true;
        if (!dyn) return t_first + it * t_step;
        const int q = it % kTaskQ2;
        bool got = mbar_wait_cluster(&m.tq_full[q], (uint32_t)(it / kTaskQ2) & 1u);
        if (warp_call) got = __all_sync(kFull, got);
        good = got;
        const int t = got ? m.tq[q] : total;
        if (warp_call) __syncwarp();
        if (got && (!warp_call || (threadIdx.x & 31) == 0)) {
            if (leader) mbar_arrive(&m.tq_empty[q]);
            else mbar_arrive_cluster(lead_tq_empty + (uint32_t)q * 8u);
        }
        return t;
    };
    const int rp = expand_rpad(a.r);
    const int apb = 64 / rp;  // adapters per expand block
    const int n_groups = a.L > 0 ? (a.L + apb - 1) / apb : 0;
    // chain row of this CTA's half for chain c of weight tile mt (chains of nu rows)
    auto chain_row = [&](int mt, int c, int nu) {
        return GATE_UP ? mt * nu + (int)rank * (nu / 2) : mt * 2 * nu + c * nu + (int)rank * (nu / 2);
    };
    // bf16 stage: byte offsets of the chain-0 rows and from them to the chain-1 rows
    auto c0_off = [&](int mode) { return mode ? kC0T : kSlot; };
    auto c1_rel = [&](int mode, int nu) { return mode ? (nu / 2) * kBK * 2 : kSlot; };
    // expand block j of a chunk's mask: the j-th adapter group with an adapter present
    auto group_present = [&](unsigned long long mask, int g) {
        const unsigned long long gm = apb >= 64 ? ~0ull : ((1ull << apb) - 1ull);
        return ((mask >> (g * apb)) & gm) != 0ull;
    };
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, armed = 0, last_par = 0;
            bool z_seen = false;
            const uint32_t full0 = cluster_addr(m.full, 0);  // the leader's full[0]
            // Take stage `stage` for copies of `bytes_pair` bytes over both CTAs
            // (counted on the leader's full barrier).  FP8 weights: this CTA's
            // `code_bytes` of codes count on its own cfull barrier; a stage
            // without codes completes its cfull phase at once, so the
            // converters walk every stage in step.
            auto acquire = [&](uint32_t bytes_pair, uint32_t code_bytes) {
                if (!mbar_wait_cluster(&m.empty[stage], phase ^ 1)) return false;
                if (leader) mbar_arrive_expect_tx(&m.full[stage], bytes_pair);
                if (W8) {
                    if (code_bytes) mbar_arrive_expect_tx(&m.cfull[stage], code_bytes);
                    else mbar_arrive(&m.cfull[stage]);
                }
                return true;
            };
            auto advance = [&]() {
                armed |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (phase << stage);
                if (++stage == NS) { stage = 0; phase ^= 1; }
            };
            // this stage's pair rows and its chain-c rows (shrink items: mode 0)
            auto xdst = [&]() { return m.ring + (size_t)stage * (W8 ? kStageW8 : kStage2); };
            auto cdst = [&](int c, int mode = 0, int nu = 0) {
                return W8 ? m.ring + (size_t)stage * kStageW8 + kC0T + c * kSlot
                          : m.ring + (size_t)stage * kStage2 + c0_off(mode) + c * c1_rel(mode, nu);
            };
            const uint32_t peer_tq = cluster_addr(m.tq, 1), peer_tq_full = cluster_addr(m.tq_full, 1);
            for (int it = 0; ok; it++) {
                int t;
                if (dyn && leader) {
                    // the next item for both CTAs: into each CTA's queue slot,
                    // once every consumer of both has read the slot's last item
                    const int q = it % kTaskQ2;
                    if (!mbar_wait(&m.tq_empty[q], (((uint32_t)(it / kTaskQ2)) & 1u) ^ 1u)) { ok = false; break; }
                    t = atomicAdd(a.task_counter, 1);
                    m.tq[q] = t;
                    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_tq + (uint32_t)q * 4u), "r"(t) : "memory");
                    mbar_arrive(&m.tq_full[q]);
                    mbar_arrive_cluster(peer_tq_full + (uint32_t)q * 8u);  // release: the store above first
                } else {
                    bool good;
                    t = take_task(it, good, false);
                    if (!good) { ok = false; break; }
                }
                if (t >= total) break;
                if (t < n_sh) {
                    // shrink item: this CTA's 128 pair rows, then the A boxes of its slots
                    ShItem sh;
                    sh.load(a, t, n_lora);
                    const int ns0 = min(sh.nb, g2), ns1 = max(0, min(sh.nb - g2, g2));
                    const int mine = rank ? ns1 : ns0, g0 = (int)rank * g2;
                    int arow[kMaxShrinkSlots / 2];
                    for (int q = 0; q < mine; q++) {
                        const int b = a.lora_buckets[sh.j0 + g0 + q];
                        arow[q] = ((b % L1 - 1) * a.E + b / L1) * a.r;  // first row of A[l][e]
                    }
                    const uint32_t bytes_pair = 2u * kSlot + (uint32_t)((ns0 + ns1) * a.r) * kBK * 2u;
                    const int rows0 = sh.q0c + (int)rank * 128;
                    const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!acquire(bytes_pair, 0u)) { ok = false; break; }
                        const uint32_t bar = full0 + (uint32_t)stage * 8u;
                        const int k0 = kb * kBK;
                        tma2_2d(xdst(), &a.xmap, bar, k0, rows0);
                        for (int q = 0; q < mine; q++)
                            tma2_2d(cdst(0) + q * a.r * kBK * 2, &a.amap, bar, k0, arow[q]);
                        advance();
                    }
                    continue;
                }
                PairTask tw;
                tw.lookup(tt, n_active, ksplit, nu0, nu1, t - n_sh);
                const int e = tw.e, nu = tw.nu, nu2 = nu / 2;
                const int rows0 = tw.q0c + (int)rank * 128;
                const int rows_t = tw.q0c + kPairRows + (int)rank * (kTailRows / 2);  // this CTA's tail rows
                const int c0row = chain_row(tw.mt, 0, nu), c1row = chain_row(tw.mt, 1, nu);
                const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
                // The task's copies, with the chunk mode and the tail fixed at
                // compile time (this thread issues every copy of its CTA; each
                // mode's maps are named directly, so the copies take the
                // parameters' own addresses).  Per CTA and stage: 128 pair rows
                // (+ 64 tail rows) + nu / 2 rows of each chain (also for expand
                // blocks); with FP8 weights the converters fill the chain rows
                // of the base K steps.
                auto produce = [&](auto M1, auto TL) {
                    constexpr bool m1 = decltype(M1)::value, tl = decltype(TL)::value;
                    const CUtensorMap* wmap = m1 ? &a.wmap_t : &a.wmap;
                    const CUtensorMap* bmap = m1 ? &a.bmap_t : &a.bmap;
                    constexpr uint32_t xbytes = (uint32_t)kSlot + (tl ? (uint32_t)kSlot / 2u : 0u);
                    const uint32_t bytes_pair = 2u * (xbytes + 2u * (uint32_t)nu2 * kBK * 2u);
                    const uint32_t bytes_base = W8 ? 2u * xbytes : bytes_pair;
                    const uint32_t code_bytes = W8 ? 2u * (uint32_t)nu2 * kBK : 0u;
                    const CUtensorMap* qmap = m1 ? &a.w8map_t : &a.w8map;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!acquire(bytes_base, code_bytes)) { ok = false; return; }
                        const uint32_t bar = full0 + (uint32_t)stage * 8u;
                        const int k0 = kb * kBK;
                        tma2_2d(xdst(), &a.xmap, bar, k0, rows0);
                        if constexpr (tl) tma2_2d(xdst() + kXTail, &a.xmap_t, bar, k0, rows_t);
                        if constexpr (W8) {
                            // this CTA's codes into the upper half of each chain's
                            // slot (the converters expand them in place)
                            uint8_t* d0 = cdst(0) + kCodeOff;
                            uint8_t* d1 = cdst(1) + kCodeOff;
                            if constexpr (GATE_UP) {
                                tma_load_4d(d0, qmap, &m.cfull[stage], k0, c0row, 0, e);
                                tma_load_4d(d1, qmap, &m.cfull[stage], k0, c0row, 1, e);
                            } else {
                                tma_load_3d(d0, qmap, &m.cfull[stage], k0, c0row, e);
                                tma_load_3d(d1, qmap, &m.cfull[stage], k0, c1row, e);
                            }
                        } else if constexpr (GATE_UP) {
                            // the gate rows, then the up rows, of this CTA's nu / 2 units
                            tma2_4d(cdst(0, m1, nu), wmap, bar, k0, c0row, 0, e);
                            tma2_4d(cdst(1, m1, nu), wmap, bar, k0, c0row, 1, e);
                        } else {
                            tma2_3d(cdst(0, m1, nu), wmap, bar, k0, c0row, e);
                            tma2_3d(cdst(1, m1, nu), wmap, bar, k0, c1row, e);
                        }
                        advance();
                    }
                    if (!expand) return;
                    const unsigned long long mask = tt.cmask[tw.chunk];
                    if (mask == 0ull) return;
                    if (!z_seen) {
                        // the expand reads zexp: every shrink item, in both CTAs of its pair, is done
                        if (!wait_count(a.zdone, 2 * n_sh_tasks)) { ok = false; return; }
                        // the shrink items' generic stores before the TMA (async proxy) reads
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        z_seen = true;
                    }
                    // expand blocks with an adapter present, dealt over the K splits
                    for (int g = 0, j = 0; g < n_groups; g++) {
                        if (!group_present(mask, g)) continue;
                        if (j++ % ksplit != tw.split) continue;
                        if (!acquire(bytes_pair, 0u)) { ok = false; return; }
                        const uint32_t bar = full0 + (uint32_t)stage * 8u;
                        const int l0 = g * apb;
                        // zexp rows of this CTA's pairs (apb adapter sub-tiles; the
                        // tail's after the main rows), then the adapters' B rows of
                        // each chain
                        tma2_3d(xdst(), &a.zxmap, bar, 0, rows0, l0);
                        if constexpr (tl) tma2_3d(xdst() + kXTail, &a.zxmap_t, bar, 0, rows_t, l0);
                        if constexpr (GATE_UP) {
                            tma2_5d(cdst(0, m1, nu), bmap, bar, 0, c0row, 0, e, l0);
                            tma2_5d(cdst(1, m1, nu), bmap, bar, 0, c0row, 1, e, l0);
                        } else {
                            tma2_4d(cdst(0, m1, nu), bmap, bar, 0, c0row, e, l0);
                            tma2_4d(cdst(1, m1, nu), bmap, bar, 0, c1row, e, l0);
                        }
                        advance();
                    }
                };
                if (tw.mode == 0) produce(BoolC<false>{}, BoolC<false>{});
                else if (tw.n_tail > 0) produce(BoolC<true>{}, BoolC<true>{});
                else produce(BoolC<true>{}, BoolC<false>{});
            }
            // every issued copy of both CTAs lands before either CTA may exit (the
            // leader's full barriers count both; the peer waits at the final
            // pair barrier)
            if (leader)
                for (int s = 0; s < NS; s++)
                    if ((armed >> s) & 1u) mbar_wait(&m.full[s], (last_par >> s) & 1u);
            // FP8 weights: and this CTA's code copies
            if (W8)
                for (int s = 0; s < NS; s++)
                    if ((armed >> s) & 1u) mbar_wait(&m.cfull[s], (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------------------- MMA issuer (leader)
            int stage = 0;
            uint32_t phase = 0;
            // descriptor bases of the stage ring; a stage adds its offset in
            // 16-byte units
            const uint64_t dxr = umma_desc_sw128(smem_u32(m.ring));
            const uint64_t dcr = dxr;
            const uint64_t exr = umma_desc_kmajor(smem_u32(m.ring), expand_layout(rp), 8u * rp * 2u);
            const uint64_t ecr = exr;
            constexpr uint64_t kSlot16 = kSlot / 16;
            constexpr uint64_t kXT16 = kXTail / 16;                       // tail rows in a stage
            constexpr uint64_t kX16 = (W8 ? kStageW8 : kStage2) / 16;    // stage stride
            constexpr uint64_t kC16 = kX16;
            const uint64_t zsub16 = 128u * rp * 2u / 16u, ztsub16 = 64u * rp * 2u / 16u;
            auto xoff = [&]() { return (uint64_t)stage * kX16; };
            auto coff = [&]() { return (uint64_t)stage * kC16; };
            // chain-0 rows within a stage, and chain 1 from chain 0
            auto c0o = [&](int md) { return W8 ? (uint64_t)kC0T / 16u : (uint64_t)c0_off(md) / 16u; };
            auto c1o = [&](int md, int nu) { return W8 ? kSlot16 : (uint64_t)c1_rel(md, nu) / 16u; };
            // a stage is ready when both CTAs' copies landed and, with FP8
            // weights, both CTAs' converters are done with it
            auto take = [&]() {
                if (!mbar_wait_cluster(&m.full[stage], phase)) return false;
                if (W8 && !mbar_wait_cluster(&m.wready[stage], phase)) return false;
                tc_fence_after();
                return true;
            };
            auto release = [&]() {
                umma2_commit_both(&m.empty[stage]);
                if (++stage == NS) { stage = 0; phase ^= 1; }
            };
            const uint32_t d_c0 = tmem_base;
            for (int it = 0; ok; it++) {
                bool good;
                const int t = take_task(it, good, false);
                if (!good) { ok = false; break; }
                if (t >= total) break;
                // the accumulator is free once both CTAs' epilogues drained the previous task
                if (!mbar_wait_cluster(m.tempty, ((uint32_t)it & 1u) ^ 1u)) { ok = false; break; }
                tc_fence_after();
                if (t < n_sh) {
                    ShItem sh;
                    sh.load(a, t, n_lora);
                    const uint32_t idesc = umma_idesc_bf16_f32(256, 256);
                    const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!take()) { ok = false; break; }
                        const uint64_t da = dxr + xoff(), db = dcr + coff() + c0o(0);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; kk++)
                            umma2_bf16(d_c0, da + 2 * kk, db + 2 * kk, idesc, (kb != kb0) || (kk != 0));
                        release();
                    }
                    if (!ok) break;
                    umma2_commit_both(m.tfull);
                    continue;
                }
                PairTask tw;
                tw.lookup(tt, n_active, ksplit, nu0, nu1, t - n_sh);
                const int nu = tw.nu, nu2 = nu / 2;
                const uint32_t idesc = umma_idesc_bf16_f32(256, nu);
                const uint32_t idesc_t = umma_idesc_bf16_f32(128, nu);
                const uint64_t bsub16 = (uint64_t)nu2 * rp * 2u / 16u;
                const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
                const unsigned long long mask = expand ? tt.cmask[tw.chunk] : 0ull;
                // The task's MMAs, with the chunk mode and the tail fixed at
                // compile time: this one thread issues every MMA of the pair,
                // and a test per MMA measurably slows the stages.
                // Accumulators: chain 0 from column 0, chain 1 from column 256
                // (mode 0) or nu (mode 1); mode-1 tails (64 lanes x nu / 2
                // columns per chain in each CTA) after both.
                auto run = [&](auto M1, auto TL) {
                    constexpr bool m1 = decltype(M1)::value, tl = decltype(TL)::value;
                    const uint32_t d_c1 = tmem_base + (m1 ? (uint32_t)nu : (uint32_t)kChain1Col);
                    const uint32_t d_t0 = tmem_base + 2u * (uint32_t)nu, d_t1 = d_t0 + (uint32_t)nu2;
                    const uint64_t c0 = c0o(m1 ? 1 : 0), c1 = m1 ? c1o(1, nu) : c1o(0, nu);
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!take()) { ok = false; return; }
                        const uint64_t da = dxr + xoff(), db = dcr + coff() + c0;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; kk++) {
                            const uint32_t acc = (kb != kb0) || (kk != 0);
                            umma2_bf16(d_c0, da + 2 * kk, db + 2 * kk, idesc, acc);
                            umma2_bf16(d_c1, da + 2 * kk, db + c1 + 2 * kk, idesc, acc);
                            if constexpr (tl) {
                                umma2_bf16(d_t0, da + kXT16 + 2 * kk, db + 2 * kk, idesc_t, acc);
                                umma2_bf16(d_t1, da + kXT16 + 2 * kk, db + c1 + 2 * kk, idesc_t, acc);
                            }
                        }
                        release();
                    }
                    for (int g = 0, j = 0; mask != 0ull && g < n_groups; g++) {
                        if (!group_present(mask, g)) continue;
                        if (j++ % ksplit != tw.split) continue;
                        if (!take()) { ok = false; return; }
                        const uint64_t ex = exr + xoff(), ec = ecr + coff() + c0;
                        for (int q = 0; q < apb; q++) {
                            const uint64_t za = ex + q * zsub16, zt = ex + kXT16 + q * ztsub16;
                            const uint64_t b0 = ec + q * bsub16, b1 = ec + c1 + q * bsub16;
                            for (int kk = 0; kk < rp / 16; kk++) {
                                umma2_bf16(d_c0, za + 2 * kk, b0 + 2 * kk, idesc, 1u);
                                umma2_bf16(d_c1, za + 2 * kk, b1 + 2 * kk, idesc, 1u);
                                if constexpr (tl) {
                                    umma2_bf16(d_t0, zt + 2 * kk, b0 + 2 * kk, idesc_t, 1u);
                                    umma2_bf16(d_t1, zt + 2 * kk, b1 + 2 * kk, idesc_t, 1u);
                                }
                            }
                        }
                        release();
                    }
                };
                if (tw.mode == 0) run(BoolC<false>{}, BoolC<false>{});
                else if (tw.n_tail > 0) run(BoolC<true>{}, BoolC<true>{});
                else run(BoolC<true>{}, BoolC<false>{});
                if (!ok) break;
                umma2_commit_both(m.tfull);
            }
        }
    } else if (W8 && warp >= kConvWarp0) {
        // ------------------------------------------------ FP8 code converters
        // Every stage of the ring, in the order the producer fills it: once
        // this CTA's codes of a base K step landed (cfull), each thread reads
        // its 16-code chunks (i = ct + 256 n: chain c, row r, chunk kc) from
        // the upper half of the chain slots, the converter warps meet at a
        // named barrier, and each writes bf16(scale x value) of its chunks in
        // the 128-byte-swizzled rows the MMA reads, over the codes' slots.
        // Stages of shrink items and expand blocks (rows by TMA) pass.  Each
        // warp then arrives on the leader's wready barrier of the stage.
        const int ct = (warp - kConvWarp0) * 32 + lane;
        const uint32_t k2p56 = pack_bf16x2(0x1p56f, 0x1p56f);
        int stage = 0;
        uint32_t phase = 0, cpar = 0;
        const uint32_t lead_wready = cluster_addr(m.wready, 0);
        // all converter threads meet (bounded); false on timeout, warp-uniform
        auto rendezvous = [&]() {
            mbar_arrive(m.cvbar);
            const bool r_ok = __all_sync(kFull, mbar_wait(m.cvbar, cpar));
            cpar ^= 1;
            return r_ok;
        };
        // waits for this stage's codes (or the producer's mark of a stage
        // without codes): the producer takes a stage only after the pair's
        // MMAs are done with its last use
        auto stage_in = [&]() { return __all_sync(kFull, mbar_wait(&m.cfull[stage], phase)); };
        auto stage_done = [&]() {
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(&m.wready[stage]);
                else mbar_arrive_cluster(lead_wready + (uint32_t)stage * 8u);
            }
            if (++stage == NS) { stage = 0; phase ^= 1; }
        };
        for (int it = 0; ok; it++) {
            bool good;
            const int t = take_task(it, good, true);
            if (!good) { ok = false; break; }
            if (t >= total) break;
            if (t < n_sh) {
                ShItem sh;
                sh.load(a, t, n_lora);
                const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                for (int kb = kb0; kb < kb1 && ok; kb++) {
                    if (!stage_in()) { ok = false; break; }
                    stage_done();
                }
                continue;
            }
            PairTask tw;
            tw.lookup(tt, n_active, ksplit, nu0, nu1, t - n_sh);
            const int nu2 = tw.nu / 2, n_chunks = 8 * nu2;
            const int c0row = chain_row(tw.mt, 0, tw.nu), c1row = chain_row(tw.mt, 1, tw.nu);
            // the factor of each of this thread's rows: bf16x2 of scale * 2^120
            // (or scale * 2^64, then 2^56, when that is beyond bf16's range)
            uint32_t fh_[4];
            bool two_[4];
#pragma unroll
            for (int n = 0; n < 4; n++) {
                const int i = ct + 256 * n;
                float sc = 0.f;
                if (i < n_chunks) {
                    const int c = i / (4 * nu2), r = (i % (4 * nu2)) >> 2;
                    if (GATE_UP) {
                        const int u = c0row + r;
                        if (u < a.I) sc = a.wscale[(size_t)tw.e * 2 * a.I + (size_t)c * a.I + u];
                    } else {
                        const int h = (c ? c1row : c0row) + r;
                        if (h < a.H) sc = a.wscale[(size_t)tw.e * a.H + h];
                    }
                }
                const float s120 = sc * 0x1p120f;
                two_[n] = !(fabsf(s120) <= 3.0e38f);
                const float f = two_[n] ? sc * 0x1p64f : s120;
                fh_[n] = pack_bf16x2(f, f);
            }
            const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
            for (int kb = kb0; kb < kb1 && ok; kb++) {
                if (!stage_in()) { ok = false; break; }
                uint8_t* slot = m.ring + (size_t)stage * kStageW8 + kC0T;
                uint4 code[4];
#pragma unroll
                for (int n = 0; n < 4; n++) {
                    const int i = ct + 256 * n;
                    if (i < n_chunks) {
                        const int c = i / (4 * nu2), rem = i % (4 * nu2), r = rem >> 2, kc = rem & 3;
                        code[n] = *reinterpret_cast<const uint4*>(slot + (size_t)c * kSlot + kCodeOff + r * kBK + kc * 16);
                    }
                }
                // every converter has its codes before any bf16 row overwrites them
                if (!rendezvous()) { ok = false; break; }
#pragma unroll
                for (int n = 0; n < 4; n++) {
                    const int i = ct + 256 * n;
                    if (i < n_chunks) {
                        const int c = i / (4 * nu2), rem = i % (4 * nu2), r = rem >> 2, kc = rem & 3;
                        uint8_t* row = slot + (size_t)c * kSlot + r * 128;
                        e4m3x16_to_bf16(code[n], fh_[n], k2p56, two_[n],
                                        reinterpret_cast<uint4*>(row + (((2 * kc) ^ (r & 7)) << 4)),
                                        reinterpret_cast<uint4*>(row + (((2 * kc + 1) ^ (r & 7)) << 4)));
                    }
                }
                // the generic stores before the tensor cores (async proxy) read them
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                stage_done();
            }
            // the expand blocks of the task (bf16 rows by TMA): only the arrival
            const unsigned long long mask = expand ? tt.cmask[tw.chunk] : 0ull;
            for (int g = 0, jj = 0; ok && mask != 0ull && g < n_groups; g++) {
                if (!group_present(mask, g)) continue;
                if (jj++ % ksplit != tw.split) continue;
                if (!stage_in()) { ok = false; break; }
                stage_done();
            }
        }
    } else {
        // -------------------------------------------------------------- epilogue
        const int ew = warp - 2;         // 0 .. kEpiWarps-1
        const int qd = warp & 3;         // TMEM lane quadrant of this warp
        const int half = ew >> 2;        // which alternate 16-column groups
        const int etid = ew * 32 + lane;
        uint32_t epar = 0;
        auto rendezvous = [&]() {
            mbar_arrive(m.ebar);
            const bool r_ok = __all_sync(kFull, mbar_wait(m.ebar, epar));
            epar ^= 1;
            return r_ok;
        };
        // the accumulator is free once both CTAs' epilogue warps released it
        const uint32_t lead_tempty = cluster_addr(m.tempty, 0);
        auto release = [&]() {
            if (leader) mbar_arrive(m.tempty);
            else mbar_arrive_cluster(lead_tempty);
        };
        const uint32_t t_lane = tmem_base + ((uint32_t)(qd * 32) << 16);
        // Column groups of 16 are drained two at a time: the TMEM loads of
        // the next group are issued before the current one is processed, so
        // their latency overlaps the arithmetic and the stores.
        //
        // gate_up: SiLU(gate) * up of 16 units into act row `arow` from unit u
        auto act_emit = [&](const uint32_t (&gr)[16], const uint32_t (&ur)[16], int u, bool row_ok, uint16_t* arow) {
            if (!row_ok) return;
            float gv[16], uv[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                gv[i] = __uint_as_float(gr[i]);
                uv[i] = __uint_as_float(ur[i]);
            }
            uint4 lo, hi;
            lo.x = pack_bf16x2(silu_fast(gv[0]) * uv[0], silu_fast(gv[1]) * uv[1]);
            lo.y = pack_bf16x2(silu_fast(gv[2]) * uv[2], silu_fast(gv[3]) * uv[3]);
            lo.z = pack_bf16x2(silu_fast(gv[4]) * uv[4], silu_fast(gv[5]) * uv[5]);
            lo.w = pack_bf16x2(silu_fast(gv[6]) * uv[6], silu_fast(gv[7]) * uv[7]);
            hi.x = pack_bf16x2(silu_fast(gv[8]) * uv[8], silu_fast(gv[9]) * uv[9]);
            hi.y = pack_bf16x2(silu_fast(gv[10]) * uv[10], silu_fast(gv[11]) * uv[11]);
            hi.z = pack_bf16x2(silu_fast(gv[12]) * uv[12], silu_fast(gv[13]) * uv[13]);
            hi.w = pack_bf16x2(silu_fast(gv[14]) * uv[14], silu_fast(gv[15]) * uv[15]);
            if (u + 8 <= a.I) *reinterpret_cast<uint4*>(arow + u) = lo;
            if (u + 16 <= a.I) *reinterpret_cast<uint4*>(arow + u + 8) = hi;
        };
        // gate_up: this warp's groups g = half, half + 2, .. < ng, gate at TMEM
        // address tg + 16 g and up at tu + 16 g, units from u0 + 16 g
        auto act_pass = [&](uint32_t tg, uint32_t tu, int u0, int ng, bool row_ok, uint16_t* arow) {
            uint32_t ga[16], ua[16], gb[16], ub[16];
            int g = half;
            if (g >= ng) return;
            if constexpr (W8) {
                // (the FP8 kernels' extra warps leave no registers for a second group)
                for (; g < ng; g += 2) {
                    tmem_ld16_issue(tg + g * 16, ga);
                    tmem_ld16_issue(tu + g * 16, ua);
                    tmem_wait_ld(ga, ua);
                    act_emit(ga, ua, u0 + g * 16, row_ok, arow);
                }
                return;
            }
            tmem_ld16_issue(tg + g * 16, ga);
            tmem_ld16_issue(tu + g * 16, ua);
            tmem_wait_ld(ga, ua);
            for (;;) {
                const int g1 = g + 2;
                if (g1 < ng) {
                    tmem_ld16_issue(tg + g1 * 16, gb);
                    tmem_ld16_issue(tu + g1 * 16, ub);
                }
                act_emit(ga, ua, u0 + g * 16, row_ok, arow);
                if (g1 >= ng) break;
                tmem_wait_ld(gb, ub);
                const int g2 = g1 + 2;
                if (g2 < ng) {
                    tmem_ld16_issue(tg + g2 * 16, ga);
                    tmem_ld16_issue(tu + g2 * 16, ua);
                }
                act_emit(gb, ub, u0 + g1 * 16, row_ok, arow);
                if (g2 >= ng) break;
                tmem_wait_ld(ga, ua);
                g = g2;
            }
        };
        // down: the pair ids and validity of the 4 rows this lane stores
        // (lane / 4 + 8 i), from the lanes that hold them
        auto store_rows = [&](int p, bool row_ok, int (&rp_row)[4], bool (&rv)[4]) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int src = (lane >> 2) + 8 * i;
                rp_row[i] = __shfl_sync(kFull, p, src);
                rv[i] = __shfl_sync(kFull, row_ok ? 1 : 0, src) != 0;
            }
        };
        // down: w * d of 16 W2 rows from h into the fp32 slab, or into the bf16
        // output when K is not split (slab null).  The warp's 32 rows x 16
        // columns go through its tile: each store then writes 64 (bf16: 32)
        // contiguous bytes of 8 rows (lane / 4 + 8 i, quarter lane % 4) instead
        // of 16 (8) bytes of 32 rows.
        float* const trw = m.tr + ew * kTrFloats;
        auto down_emit = [&](const uint32_t (&vr)[16], float* slab, int h, float w, const int (&rp_row)[4],
                             const bool (&rv)[4]) {
            float4* mine = reinterpret_cast<float4*>(trw + lane * kTrStride);
#pragma unroll
            for (int j = 0; j < 4; j++)
                mine[j] = make_float4(w * __uint_as_float(vr[4 * j]), w * __uint_as_float(vr[4 * j + 1]),
                                      w * __uint_as_float(vr[4 * j + 2]), w * __uint_as_float(vr[4 * j + 3]));
            __syncwarp();
            const int c4 = lane & 3;
            const int hh = h + 4 * c4;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int row = (lane >> 2) + 8 * i;
                const float4 val = *reinterpret_cast<const float4*>(trw + row * kTrStride + 4 * c4);
                if (rv[i] && hh + 4 <= a.H) {
                    if (slab) {
                        *reinterpret_cast<float4*>(slab + (size_t)rp_row[i] * a.H + hh) = val;
                    } else {
                        const uint2 o = make_uint2(pack_bf16x2(val.x, val.y), pack_bf16x2(val.z, val.w));
                        *reinterpret_cast<uint2*>(a.pair_out16 + (size_t)rp_row[i] * a.H + hh) = o;
                    }
                }
            }
            __syncwarp();
        };
        // down: this warp's groups g = half, half + 2, .. < ng at TMEM address
        // t0 + 16 g, W2 rows from h0 + 16 g
        auto down_pass = [&](float* slab, uint32_t t0, int h0, int ng, float w, const int (&rp_row)[4],
                             const bool (&rv)[4]) {
            uint32_t va[16], vb[16];
            int g = half;
            if (g >= ng) return;
            if constexpr (W8) {
                for (; g < ng; g += 2) {
                    tmem_ld16_issue(t0 + g * 16, va);
                    tmem_wait_ld(va);
                    down_emit(va, slab, h0 + g * 16, w, rp_row, rv);
                }
                return;
            }
            tmem_ld16_issue(t0 + g * 16, va);
            tmem_wait_ld(va);
            for (;;) {
                const int g1 = g + 2;
                if (g1 < ng) tmem_ld16_issue(t0 + g1 * 16, vb);
                down_emit(va, slab, h0 + g * 16, w, rp_row, rv);
                if (g1 >= ng) break;
                tmem_wait_ld(vb);
                const int g2 = g1 + 2;
                if (g2 < ng) tmem_ld16_issue(t0 + g2 * 16, va);
                down_emit(vb, slab, h0 + g1 * 16, w, rp_row, rv);
                if (g2 >= ng) break;
                tmem_wait_ld(va);
                g = g2;
            }
        };
        for (int it = 0; ok; it++) {
            bool good;
            const int t = take_task(it, good, true);
            if (!good) { ok = false; break; }
            if (t >= total) break;
            if (t < n_sh) {
                if (!shrink_epilogue_m(a, t, n_lora, it, tmem_base, qd, half, lane, etid, m, rendezvous, release,
                                       (int)rank)) {
                    ok = false;
                    break;
                }
                continue;
            }
            PairTask tw;
            tw.lookup(tt, n_active, ksplit, nu0, nu1, t - n_sh);
            const int nu = tw.nu, nu2 = nu / 2;
            // accumulator columns: chain 1 from c1col; mode-1 tails from tcol
            // (chain c at tcol + c * nu / 2)
            const uint32_t c1col = tw.mode ? (uint32_t)nu : (uint32_t)kChain1Col;
            const uint32_t tcol = 2u * (uint32_t)nu;
            // this lane's main pair row of the chunk
            const int row = (int)rank * 128 + qd * 32 + lane;
            const bool valid = row < tw.n_main;
            const size_t q = (size_t)tw.q0c + row;
            // mode-1 tail: TMEM lane qd * 32 + lane holds tail row (qd % 2) * 32
            // + lane of this CTA's 64 and the half qd / 2 of each chain's columns
            const bool tail = tw.n_tail > 0;
            const int rt = (int)rank * (kTailRows / 2) + (qd & 1) * 32 + lane;
            const bool valid_t = tail && rt < tw.n_tail;
            const size_t qt = (size_t)tw.q0c + kPairRows + rt;
            const int hc = qd >> 1;
            int p = 0, pt = 0;
            float w = 0.f, wt = 0.f;
            if (!GATE_UP) {
                if (valid) {
                    p = a.compact_ids[q];
                    w = a.topk_weights[p];
                }
                if (valid_t) {
                    pt = a.compact_ids[qt];
                    wt = a.topk_weights[pt];
                }
            }
            // warp-uniform: the TMEM loads below are warp-collective
            if (!__all_sync(kFull, mbar_wait(m.tfull, (uint32_t)it & 1u))) { ok = false; break; }
            tc_fence_after();
            if (GATE_UP) {
                // units u0 + 16 g ..: gate in columns 16 g.., up c1col further
                const int u0 = tw.mt * nu;
                act_pass(t_lane, t_lane + c1col, u0, nu / 16, valid, a.act_out + q * a.I);
                // tail lanes: units u0 + hc * nu / 2 + 16 g .. of their row
                if (tail)
                    act_pass(t_lane + tcol, t_lane + tcol + nu2, u0 + hc * nu2, nu2 / 16, valid_t, a.act_out + qt * a.I);
            } else {
                // W2 rows h0 + c * nu + 16 g ..: w * d into this split's fp32 slab
                // of pair_out, or (no K split) into the bf16 pair_out16
                float* const slab = ksplit > 1 ? a.pair_out + (size_t)tw.split * a.pair_split : nullptr;
                int rp_row[4];
                bool rv[4];
                store_rows(p, valid, rp_row, rv);
                for (int c = 0; c < 2; c++)
                    down_pass(slab, t_lane + c * c1col, tw.mt * 2 * nu + c * nu, nu / 16, w, rp_row, rv);
                if (tail) {
                    store_rows(pt, valid_t, rp_row, rv);
                    for (int c = 0; c < 2; c++)
                        down_pass(slab, t_lane + tcol + c * nu2, tw.mt * 2 * nu + c * nu + hc * nu2, nu2 / 16, wt,
                                  rp_row, rv);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
    }

    if (!ok) atomicOr(&a.hdr->status, kStatusTimeout);
    // all roles of both CTAs done (every wait above is bounded): release TMEM
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc2(tmem_base, kTmem2);
}

template <bool G, bool W8>
cudaError_t set_attr2() {
    return cudaFuncSetAttribute(k_moe_gemm_2sm<G, W8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemLimit);
}

template <bool G, bool W8>
int max_pairs_of() {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(W8 ? kThreadsW8 : kTcThreads);
    cfg.dynamicSmemBytes = kTcSmemLimit;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_moe_gemm_2sm<G, W8>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

// at least half an SM's shared memory: one CTA per SM, so the whole TMEM
// allocation never waits for another CTA
// (nstages stages of kStageW8 with FP8 weights, else of kStage2)
int tc2_smem_bytes(int E, int nstages, int max_chunks, bool w8) {
    const int rings = nstages * (w8 ? kStageW8 : kStage2);
    const int bars = (2 * nstages + (w8 ? 2 * nstages : 0) + 4 + 2 * kTaskQ2) * 8 + 16 + kTaskQ2 * 4;
    const int slots = (3 * kMaxShrinkSlots + 4) * 4;
    const int table = 8 * max_chunks + (6 * E + 2) * 4;
    const int tr = 16 + kEpiWarps * kTrFloats * 4;
    return std::max(1024 + rings + bars + slots + table + tr, kTcSmemLimit / 2 + 1024);
}

int tc2_plan_stages(int E, int max_chunks) {
    for (int ns = 8; ns >= 3; ns--)
        if (tc2_smem_bytes(E, ns, max_chunks, false) <= kTcSmemLimit) return ns;
    return 0;
}

// FP8 weights: the deepest ring of 56 KiB stages that fits (at least two)
int tc2_plan_stages_w8(int E, int max_chunks) {
    for (int ns = 8; ns >= 2; ns--)
        if (tc2_smem_bytes(E, ns, max_chunks, true) <= kTcSmemLimit) return ns;
    return 0;
}

cudaError_t init_tc2_attributes() {
    cudaError_t e;
    if ((e = set_attr2<true, false>()) != cudaSuccess) return e;
    if ((e = set_attr2<false, false>()) != cudaSuccess) return e;
    if ((e = set_attr2<true, true>()) != cudaSuccess) return e;
    return set_attr2<false, true>();
}

// Pairs of this kernel that fit on the device at once (with the largest
// shared-memory request; the FP8 kernels have one more warp): the persistent
// grid must not exceed it, since tasks wait on each other's progress (shrink
// before expand).
int tc2_max_pairs(bool gate_up) {
    const int a = gate_up ? max_pairs_of<true, false>() : max_pairs_of<false, false>();
    const int b = gate_up ? max_pairs_of<true, true>() : max_pairs_of<false, true>();
    return std::min(a, b);
}

// grid: an even number of CTAs (pairs of SMs); clusters of two, with the
// programmatic-dependent-launch attribute when asked
cudaError_t launch_moe_gemm_2sm(const TcArgs& args, bool gate_up, int grid, cudaStream_t stream, bool pdl) {
    if (args.nu < 16 || args.nu > 256 || args.nu % 16 != 0) return cudaErrorInvalidValue;
    if (args.nu_t != 0 && (args.nu_t < 32 || args.nu_t > 160 || args.nu_t % 32 != 0)) return cudaErrorInvalidValue;
    if (args.r > 0 && (128 / args.r) * 2 > kMaxShrinkSlots) return cudaErrorInvalidValue;
    if (args.w8 && (args.nstages < 2 || args.wscale == nullptr)) return cudaErrorInvalidValue;
    const int smem = tc2_smem_bytes(args.E, args.nstages, args.max_chunks, args.w8 != 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(args.w8 ? kThreadsW8 : kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int n = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (args.w8) {
        if (gate_up) return cudaLaunchKernelEx(&cfg, k_moe_gemm_2sm<true, true>, args);
        return cudaLaunchKernelEx(&cfg, k_moe_gemm_2sm<false, true>, args);
    }
    if (gate_up) return cudaLaunchKernelEx(&cfg, k_moe_gemm_2sm<true, false>, args);
    return cudaLaunchKernelEx(&cfg, k_moe_gemm_2sm<false, false>, args);
}

}  // namespace moelora
