// moe_gemm_2sm.cu -- the grouped expert GEMMs for wide pair chunks (prefill
// and other many-pairs-per-expert batches) on a CTA pair: one
// tcgen05.mma.cta_group::2 with M = 256 weight rows, the pair's two CTAs
// holding 128 rows each, and N up to 128 (gate_up) or 256 (down) pairs, each
// CTA holding half of the pair rows.  Per unit of work a CTA stages half the
// pair rows of the single-CTA kernel.  It is selected by MOELORA_OPT_PAIR_CTA
// only: on the prefill workload it measured no faster than the single-CTA
// kernel (its stages move about as many shared-memory bytes per MMA, and its
// 256-unit gate_up tiles waste more of a ragged intermediate size).
//
// Layer math ("Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Implementing multi-LoRA
// inference for MoE models in vLLM", Figure 1), per routed pair:
//   gate_up:  g = W1[e] x + B1[l][e] z1,  act = SiLU(g[0:I]) * g[I:2I]
//   down:     d = W2[e] act + B2[l][e] z2, pair_out = w * d
//
// A task is (active expert, weight tile, pair chunk): gate_up chunks of at
// most 128 pairs, down chunks of at most 256.  The gate_up tile is 256
// intermediate units: the CTA of rank q holds the gate rows and the up rows
// of units 128q .. 128q+127 and the pair issues two MMAs per K step, one into
// a gate and one into an up accumulator (independent chains, so one's MMA
// latency overlaps the other's; the gate and up values of a unit land in the
// same TMEM lane, 128 columns apart).  The down tile is 256 rows of W2, 128
// per CTA.  Both GEMMs keep two accumulator sets of 256 columns, so one
// task's epilogue overlaps the next task's MMAs.  LoRA shrink items stack the A
// matrices of up to 2 * 128 / r adapter buckets on M (128 / r per CTA), and
// the expand blocks are extra K-blocks (B rows of the chunk's adapters x
// zexp rows), as in the single-CTA kernel.
//
// Roles, in each CTA of the pair (one pair per two SMs, persistent, tasks
// dealt round-robin over the pairs):
//   warp 0   TMA producer for this CTA's halves of every stage; the copies
//            of both CTAs count on the leader's (rank 0) full barrier
//            (.cta_group::2 copies), which the leader arms with both byte
//            counts;
//   warp 1   allocates TMEM (collectively with the peer); in the leader one
//            thread issues every MMA of the pair and commits stage releases
//            and accumulator completion to both CTAs' mbarriers;
//   warps 2-9 epilogue of this CTA's 128 TMEM lanes; the peer's epilogue
//            warps free an accumulator set on the leader's mbarrier.
// Every wait is bounded; on a timeout the CTA records kStatusTimeout, keeps
// walking its loops without waiting (so its peer is never left waiting on
// it), drains its copies, frees TMEM and exits.
#include "gemm_tasks.cuh"

namespace moelora {

namespace {

constexpr int kPairBN = 256;                     // most pairs in a chunk or shrink item (column staging)
constexpr int kTmem2 = 512;                      // the whole TMEM of the SM
constexpr int kMaxNAcc2 = 2;
constexpr int kSub = 64 * kBK * 2;               // one 64-row box of pair rows (8 KiB)

template <bool GATE_UP>
struct Pair {
    // pairs per chunk: gate_up 128 (its gate and up accumulators of N <= 128
    // fill 256 columns, so two accumulator sets fit), down 256
    static constexpr int kBN = GATE_UP ? 128 : 256;
    // weight bytes per stage: gate_up the CTA's 128 gate rows and their 128
    // up rows, down its 128 W2 rows; then this CTA's half of the pair rows
    // in 64-row boxes
    static constexpr int kW = GATE_UP ? 2 * kATile : kATile;
    static constexpr int kStage = kW + (kBN / 128) * kSub;
    static constexpr int kAccCols = 256;             // TMEM columns per accumulator set
    static constexpr int kNAcc = kTmem2 / kAccCols;  // 2: one task's epilogue overlaps the next task's MMAs
};

// MMA N of a chunk: pairs rounded up to 32, so each CTA holds a multiple of 16 rows
__device__ __forceinline__ int n32(int n_real) { return (n_real + 31) & ~31; }

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

// Shared memory after the stage ring: column staging, verdicts, barriers,
// the TMEM base and the task table.
struct Smem2 {
    uint8_t* ring;
    int* s_pair;      // [kPairBN] pair id of each column (shrink items: slot column ranges)
    int* s_lora;      // [kPairBN]
    float* s_w;       // [kPairBN] top-k weight of each column
    int* s_misc;      // [kMisc]
    uint64_t* full;   // [NS] leader: both CTAs' copies of stage s landed
    uint64_t* empty;  // [NS] the pair's MMAs are done with stage s
    uint64_t* tfull;  // [kNAcc] accumulator set ready for the epilogue
    uint64_t* tempty; // [kNAcc] leader: accumulator set drained by both CTAs' epilogues
    uint64_t* ebar;   // epilogue rendezvous
    uint32_t* tmem_slot;
    TaskTable tt;
};

__device__ inline Smem2 carve2(uint8_t* base, const TcArgs& a, int NS, int stage_bytes) {
    Smem2 m;
    m.ring = base;
    uint8_t* p = base + (size_t)NS * stage_bytes;
    m.s_pair = reinterpret_cast<int*>(p);
    m.s_lora = m.s_pair + kPairBN;
    m.s_w = reinterpret_cast<float*>(m.s_lora + kPairBN);
    m.s_misc = reinterpret_cast<int*>(m.s_w + kPairBN);
    uint64_t* bars = reinterpret_cast<uint64_t*>(m.s_misc + kMisc + (kMisc & 1));
    m.full = bars;
    m.empty = m.full + NS;
    m.tfull = m.empty + NS;
    m.tempty = m.tfull + kMaxNAcc2;
    m.ebar = m.tempty + kMaxNAcc2;
    m.tmem_slot = reinterpret_cast<uint32_t*>(m.ebar + 1);
    m.tt.cmask = reinterpret_cast<unsigned long long*>(m.tmem_slot + 4);
    m.tt.e = reinterpret_cast<int*>(m.tt.cmask + a.max_chunks);
    m.tt.q0 = m.tt.e + a.E;
    m.tt.m = m.tt.q0 + a.E;
    m.tt.cum = m.tt.m + a.E;
    return m;
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kTcThreads, 1) k_moe_gemm_2sm(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int NS = a.nstages;
    using PT = Pair<GATE_UP>;
    Smem2 m = carve2(base, a, NS, PT::kStage);
    const TaskTable& tt = m.tt;
    const uint32_t rank = cta_rank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
        }
        for (int b = 0; b < PT::kNAcc; b++) {
            mbar_init(&m.tfull[b], 1);
            mbar_init(&m.tempty[b], 2 * kEpiWarps);
        }
        mbar_init(m.ebar, kEpiWarps * 32);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc2(m.tmem_slot, kTmem2);
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&a.wmap);
        prefetch_tensormap(&a.xmap);
        if (a.sh_tasks) prefetch_tensormap(&a.amap);
        if (a.tc_expand) {
            prefetch_tensormap(&a.bmap1);
            prefetch_tensormap(&a.zxmap1);
        }
    }
    tc_fence_before();
    __syncthreads();
    // the peer's barriers exist before any arrival crosses the pair
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *m.tmem_slot;

    pdl_wait();
    pdl_trigger();

    // weight tiles: 256 units (gate_up) or W2 rows (down), 128 per CTA
    const int N_out = GATE_UP ? a.I : a.H;
    const int K = GATE_UP ? a.H : a.I;
    const int ntiles = (N_out + 255) / 256;
    const int nkb = (K + kBK - 1) / kBK;
    const int n_active = a.hdr->n_active;
    build_task_table<PT::kBN>(a, tt, n_active, ntiles);
    const int ksplit = a.ksplit;
    const bool shrink = a.sh_tasks != nullptr && a.r > 0;
    const bool expand = a.tc_expand != 0 && a.r > 0;
    const int sh_ks = a.sh_ks;
    const int n_sh_tasks = shrink ? a.hdr->n_shrink_tasks : 0;
    const int n_sh = n_sh_tasks * sh_ks;
    const int n_lora = shrink ? a.hdr->n_lora_buckets : 0;
    const int L1 = a.L + 1;
    const int g_cta = a.r > 0 ? 128 / a.r : 0;  // shrink slots per CTA
    const int total = n_sh + tt.cum[n_active] * ksplit;
    const int t_first = (int)cluster_index(), t_step = (int)cluster_count();
    const int rp = expand_rpad(a.r);
    const uint32_t xa1 = 128u * rp * 2u;  // one adapter's weight-row sub-tile (and down's zexp sub-tile)
    // one adapter's zexp sub-tile (this CTA's half of the chunk's pairs)
    const uint32_t zx1 = (uint32_t)(PT::kBN / 2) * rp * 2u;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // This CTA's halves of every stage: its 128 weight (or adapter) rows and
        // its half of the chunk's pair rows, in 64-row boxes.  The copies count
        // on the leader's full barrier; the leader arms it with both CTAs' bytes.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, armed = 0, last_par = 0;
            bool z_seen = false;
            const uint32_t full0 = cluster_addr(m.full, 0);  // the leader's full[0]
            // wait until the pair's MMAs are done with the slot; the leader arms it
            auto acquire = [&](uint32_t bytes_pair) {
                if (!mbar_wait_cluster(&m.empty[stage], phase ^ 1)) return false;
                if (leader) mbar_arrive_expect_tx(&m.full[stage], bytes_pair);
                return true;
            };
            auto advance = [&]() {
                armed |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (phase << stage);
                if (++stage == NS) { stage = 0; phase ^= 1; }
            };
            for (int t = t_first; t < total && ok; t += t_step) {
                if (t < n_sh) {
                    // shrink item: this CTA's slots' A boxes, then its half of the pair rows
                    ShItem sh;
                    sh.load(a, t, n_lora);
                    const int ns0 = max(0, min(sh.nb, g_cta)), ns1 = max(0, min(sh.nb - g_cta, g_cta));
                    const int g0 = (int)rank * g_cta, ns_mine = rank ? ns1 : ns0;
                    int arow[kMaxSlots];
                    for (int q = 0; q < ns_mine; q++) {
                        const int b = a.lora_buckets[sh.j0 + g0 + q];
                        arow[q] = ((b % L1 - 1) * a.E + b / L1) * a.r;  // first row of A[l][e]
                    }
                    const int half = n32(sh.n_real) / 2, n_box = (half + 63) / 64;
                    const int brow0 = sh.q0c + (int)rank * half;
                    const uint32_t bytes_pair = (uint32_t)((ns0 + ns1) * a.r + 2 * n_box * 64) * kBK * 2;
                    const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!acquire(bytes_pair)) { ok = false; break; }
                        uint8_t* dst = m.ring + (size_t)stage * PT::kStage;
                        const uint32_t bar = full0 + (uint32_t)stage * 8u;
                        const int k0 = kb * kBK;
                        for (int q = 0; q < ns_mine; q++) tma2_2d(dst + q * a.r * kBK * 2, &a.amap, bar, k0, arow[q]);
                        for (int g = 0; g < n_box; g++)
                            tma2_2d(dst + kATile + g * 64 * kBK * 2, &a.xmap, bar, k0, brow0 + g * 64);
                        advance();
                    }
                    continue;
                }
                Task<PT::kBN> tw;
                tw.lookup(tt, n_active, ksplit, ntiles, t - n_sh);
                // this CTA's half of the chunk's pair rows (N = pairs rounded up
                // to 32), in 64-row boxes
                const int e = tw.e, half = n32(tw.n_real) / 2, n_box = (half + 63) / 64;
                const int brow0 = tw.q0c + (int)rank * half;
                // first of this CTA's 128 units (gate_up) or W2 rows (down)
                const int wrow0 = tw.mt * 256 + (int)rank * 128;
                const uint32_t bytes_pair = 2u * ((uint32_t)PT::kW + (uint32_t)n_box * kSub);
                const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
                ExpandRange xr;
                xr.none();
                int n_x = 0;
                if (expand) {
                    xr.from_mask(a, tt.cmask[tw.chunk], tw.split, ksplit);
                    n_x = xr.count();
                }
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!acquire(bytes_pair)) { ok = false; break; }
                    uint8_t* dst = m.ring + (size_t)stage * PT::kStage;
                    const uint32_t bar = full0 + (uint32_t)stage * 8u;
                    const int k0 = kb * kBK;
                    if (GATE_UP) {
                        // the gate rows of the CTA's 128 units, then their up rows
                        tma2_4d(dst, &a.wmap, bar, k0, wrow0, 0, e);
                        tma2_4d(dst + kATile, &a.wmap, bar, k0, wrow0, 1, e);
                    } else {
                        tma2_3d(dst, &a.wmap, bar, k0, wrow0, e);
                    }
                    for (int g = 0; g < n_box; g++) tma2_2d(dst + PT::kW + g * kSub, &a.xmap, bar, k0, brow0 + g * 64);
                    advance();
                }
                if (ok && n_x > 0 && !z_seen) {
                    // the expand reads zexp: every shrink item, in both CTAs of its pair, is done
                    if (!wait_count(a.zdone, 2 * n_sh_tasks)) ok = false;
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    z_seen = true;
                }
                // packed expand blocks: the next 64 / r_pad adapters present in the
                // chunk; per adapter this CTA's 128 B rows and its zexp rows
                unsigned long long rem = n_x > 0 ? xr.bits : 0ull;
                for (int g = 0, mine = xr.split; ok && rem != 0ull; g++) {
                    if (g != mine) {
                        for (int q = 0; q < xr.apb; q++) rem &= rem - 1ull;
                        continue;
                    }
                    mine += xr.ksplit;
                    int ids[4];
                    int cnt = 0;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        if (q < xr.apb && rem != 0ull) {
                            ids[q] = __ffsll((long long)rem) - 1;
                            rem &= rem - 1ull;
                            cnt = q + 1;
                        }
                    }
                    // per adapter and CTA: B rows (gate_up: gate and up sub-tiles) and zexp rows
                    if (!acquire((uint32_t)cnt * 2u * ((GATE_UP ? 2u : 1u) * xa1 + zx1))) { ok = false; break; }
                    uint8_t* dst = m.ring + (size_t)stage * PT::kStage;
                    const uint32_t bar = full0 + (uint32_t)stage * 8u;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        if (q < cnt) {
                            if (GATE_UP) {
                                // coordinates (k, unit, half, expert, adapter)
                                tma2_5d(dst + q * xa1, &a.bmap1, bar, 0, wrow0, 0, e, ids[q]);
                                tma2_5d(dst + kATile + q * xa1, &a.bmap1, bar, 0, wrow0, 1, e, ids[q]);
                            } else {
                                tma2_4d(dst + q * xa1, &a.bmap1, bar, 0, wrow0, e, ids[q]);
                            }
                            tma2_3d(dst + PT::kW + q * zx1, &a.zxmap1, bar, 0, brow0, ids[q]);
                        }
                    }
                    advance();
                }
            }
            // every issued copy of both CTAs lands before either CTA may exit (the
            // leader's full barriers count both; the peer waits at the final
            // cluster barrier)
            if (leader)
                for (int s = 0; s < NS; s++)
                    if ((armed >> s) & 1u) mbar_wait(&m.full[s], (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------------------- MMA issuer (leader)
            // Walks the same items as the producers; a stage is used once both
            // CTAs' copies landed (the leader's full barrier counts both); its
            // release and each accumulator's completion are committed to the
            // barriers of both CTAs.
            int stage = 0;
            uint32_t phase = 0;
            const uint32_t xa16 = xa1 / 16, zx16 = zx1 / 16;
            const uint64_t d0 = umma_desc_sw128(smem_u32(m.ring));
            const uint64_t dx0 = umma_desc_kmajor(smem_u32(m.ring), expand_layout(rp), 8u * rp * 2u);
            constexpr uint64_t kStage16 = PT::kStage / 16, kA16 = kATile / 16, kW16 = PT::kW / 16;
            auto take = [&]() {
                if (!mbar_wait_cluster(&m.full[stage], phase)) return false;
                tc_fence_after();
                return true;
            };
            auto release = [&]() {
                umma2_commit_both(&m.empty[stage]);
                if (++stage == NS) { stage = 0; phase ^= 1; }
            };
            for (int t = t_first, it = 0; t < total && ok; t += t_step, it++) {
                const int b = it % PT::kNAcc;
                if (!mbar_wait_cluster(&m.tempty[b], ((uint32_t)(it / PT::kNAcc) & 1u) ^ 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(b * PT::kAccCols);
                if (t < n_sh) {
                    ShItem sh;
                    sh.load(a, t, n_lora);
                    const uint32_t idesc = umma_idesc_bf16_f32(256, n32(sh.n_real));
                    const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!take()) { ok = false; break; }
                        const uint64_t da = d0 + (uint64_t)stage * kStage16;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; kk++)
                            umma2_bf16(d, da + 2 * kk, da + kA16 + 2 * kk, idesc, (kb != kb0) || (kk != 0));
                        release();
                    }
                    if (!ok) break;
                    umma2_commit_both(&m.tfull[b]);
                    continue;
                }
                Task<PT::kBN> tw;
                tw.lookup(tt, n_active, ksplit, ntiles, t - n_sh);
                // gate_up: a gate and an up chain per K step (independent
                // accumulators, so one's MMA latency overlaps the other's)
                const uint32_t idesc = umma_idesc_bf16_f32(256, n32(tw.n_real));
                const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!take()) { ok = false; break; }
                    const uint64_t da = d0 + (uint64_t)stage * kStage16;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; kk++) {
                        const uint32_t acc = (kb != kb0) || (kk != 0);
                        umma2_bf16(d, da + 2 * kk, da + kW16 + 2 * kk, idesc, acc);
                        if (GATE_UP) umma2_bf16(d + PT::kBN, da + kA16 + 2 * kk, da + kW16 + 2 * kk, idesc, acc);
                    }
                    release();
                }
                if (ok && expand) {
                    ExpandRange xr;
                    xr.from_mask(a, tt.cmask[tw.chunk], tw.split, ksplit);
                    const int ng = xr.groups();
                    for (int g = xr.split; g < ng && ok; g += xr.ksplit) {
                        const int cnt = xr.group_size(g);
                        if (!take()) { ok = false; break; }
                        const uint64_t dxs = dx0 + (uint64_t)stage * kStage16;
                        for (int q = 0; q < cnt; q++) {
                            const uint64_t da = dxs + q * xa16, db = dxs + kW16 + q * zx16;
                            for (int kk = 0; kk < rp / 16; kk++) {
                                umma2_bf16(d, da + 2 * kk, db + 2 * kk, idesc, 1u);
                                if (GATE_UP) umma2_bf16(d + PT::kBN, da + kA16 + 2 * kk, db + 2 * kk, idesc, 1u);
                            }
                        }
                        release();
                    }
                }
                if (!ok) break;
                umma2_commit_both(&m.tfull[b]);
            }
        }
    } else {
        // -------------------------------------------------------------- epilogue
        const int ew = warp - 2;         // 0 .. kEpiWarps-1
        const int qd = warp & 3;         // TMEM lane quadrant of this warp
        const int half = ew >> 2;        // which alternate 16-column chunks
        const int etid = ew * 32 + lane;
        uint32_t epar = 0;
        auto rendezvous = [&]() {
            mbar_arrive(m.ebar);
            const bool r_ok = __all_sync(kFull, mbar_wait(m.ebar, epar));
            epar ^= 1;
            return r_ok;
        };
        // an accumulator set is free once both CTAs' epilogue warps released it
        const uint32_t lead_tempty = cluster_addr(m.tempty, 0);
        auto release = [&](int bb) {
            if (leader) mbar_arrive(&m.tempty[bb]);
            else mbar_arrive_cluster(lead_tempty + (uint32_t)bb * 8u);
        };
        for (int t = t_first, it = 0; t < total && ok; t += t_step, it++) {
            const int b = it % PT::kNAcc;
            const int use = it / PT::kNAcc;
            if (t < n_sh) {
                if (!shrink_epilogue(a, t, n_lora, b, use, tmem_base, PT::kAccCols, qd, half, lane, etid, m.s_pair,
                                     m.s_lora, m.s_misc, m.tfull, rendezvous, release, (int)rank, 2)) {
                    ok = false;
                    break;
                }
                continue;
            }
            Task<PT::kBN> tw;
            tw.lookup(tt, n_active, ksplit, ntiles, t - n_sh);
            const int q0c = tw.q0c, n_real = tw.n_real;
            // stage the column data while the task's MMAs run (after everyone is
            // done with the previous task's)
            if (!rendezvous()) { ok = false; break; }
            for (int c = etid; c < n_real; c += kEpiWarps * 32) {
                const int p = a.compact_ids[q0c + c];
                m.s_pair[c] = p;
                m.s_w[c] = a.topk_weights[p];
            }
            if (!rendezvous()) { ok = false; break; }
            // warp-uniform: the TMEM loads below are warp-collective
            const bool got = __all_sync(kFull, mbar_wait(&m.tfull[b], (uint32_t)use & 1u));
            tc_fence_after();
            const uint32_t t_lane = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(b * PT::kAccCols);
            bool step_ok = got;
            if (GATE_UP) {
                // lane = one of this CTA's 128 units; its gate values in columns
                // 0..127 and its up values 128 columns further
                const int w_unit = tw.mt * 256 + (int)rank * 128 + qd * 32 + lane;
                for (int c0 = half * 16; got && c0 < n_real; c0 += 32) {
                    float g[16], u[16];
                    tmem_ld16x2(t_lane + c0, t_lane + PT::kBN + c0, g, u);
                    if (w_unit < a.I) {
#pragma unroll
                        for (int c = 0; c < 16; c++) {
                            const int cc = c0 + c;
                            if (cc < n_real)
                                a.act_out[(size_t)(q0c + cc) * a.I + w_unit] = f32_to_bf16_rne(silu_fast(g[c]) * u[c]);
                        }
                    }
                }
            } else {
                // this CTA's 128 W2 rows; with split K every split writes its own slab
                const int w_row = tw.mt * 256 + (int)rank * 128 + qd * 32 + lane;
                float* const pout = a.pair_out + (ksplit > 1 ? (size_t)tw.split * a.pair_split : 0);
                for (int c0 = half * 16; got && c0 < n_real; c0 += 32) {
                    float g[16];
                    tmem_ld16(t_lane + c0, g);
                    if (w_row < a.H) {
#pragma unroll
                        for (int c = 0; c < 16; c++) {
                            const int cc = c0 + c;
                            if (cc < n_real) pout[(size_t)m.s_pair[cc] * a.H + w_row] = m.s_w[cc] * g[c];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(b);
            if (!step_ok) { ok = false; break; }
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

template <bool G>
cudaError_t set_attr2() {
    return cudaFuncSetAttribute(k_moe_gemm_2sm<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemLimit);
}

}  // namespace

// at least half an SM's shared memory: one CTA per SM, so the whole TMEM
// allocation never waits for another CTA
int tc2_smem_bytes(bool gate_up, int E, int nstages, int max_chunks) {
    const int stage = gate_up ? Pair<true>::kStage : Pair<false>::kStage;
    const int staging = 3 * kPairBN * 4 + (kMisc + (kMisc & 1)) * 4;
    const int bars = (2 * nstages + 2 * kMaxNAcc2 + 1) * 8 + 16;
    const int table = 8 * max_chunks + (4 * E + 1) * 4;
    return std::max(1024 + nstages * stage + staging + bars + table, kTcSmemLimit / 2 + 1024);
}

int tc2_plan_stages(bool gate_up, int E, int max_chunks) {
    for (int ns = 8; ns >= 3; ns--)
        if (tc2_smem_bytes(gate_up, E, ns, max_chunks) <= kTcSmemLimit) return ns;
    return 0;
}

cudaError_t init_tc2_attributes() {
    cudaError_t e;
    if ((e = set_attr2<true>()) != cudaSuccess) return e;
    return set_attr2<false>();
}

// Pairs of this kernel that fit on the device at once (with the largest
// shared-memory request): the persistent grid must not exceed it, since items
// wait on each other's progress (shrink before expand).
int tc2_max_pairs(bool gate_up) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmemLimit;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = gate_up ? cudaOccupancyMaxActiveClusters(&n, k_moe_gemm_2sm<true>, &cfg)
                                  : cudaOccupancyMaxActiveClusters(&n, k_moe_gemm_2sm<false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// grid: an even number of CTAs (pairs of SMs); clusters of two, with the
// programmatic-dependent-launch attribute when asked
cudaError_t launch_moe_gemm_2sm(const TcArgs& args, bool gate_up, int grid, cudaStream_t stream, bool pdl) {
    const int smem = tc2_smem_bytes(gate_up, args.E, args.nstages, args.max_chunks);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
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
    if (gate_up) return cudaLaunchKernelEx(&cfg, k_moe_gemm_2sm<true>, args);
    return cudaLaunchKernelEx(&cfg, k_moe_gemm_2sm<false>, args);
}

}  // namespace moelora
