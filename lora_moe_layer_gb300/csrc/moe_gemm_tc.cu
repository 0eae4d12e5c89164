// moe_gemm_tc.cu -- the grouped expert GEMMs on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), with the LoRA expand and the activation or
// top-k weight in the epilogue.
//
// Layer math ("Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Implementing multi-LoRA
// inference for MoE models in vLLM", Figure 1), per routed pair:
//   gate_up:  g = W1[e] x + B1[l][e] z1,  act = SiLU(g[0:I]) * g[I:2I]
//   down:     d = W2[e] act + B2[l][e] z2, pair_out = w * d
//
// Operand order follows the swap-AB idea of the fused-MoE news item (its
// first optimisation): the long weight dimension goes on the MMA's M side
// (128 weight rows per task) and the expert's pairs on N (16..BN columns), so
// a decode step with two or three pairs per expert still issues full-height
// MMAs, and a prefill chunk fills N up to BN.  A task is (active expert,
// 128-row weight tile, chunk of at most BN pairs).
//
// The LoRA shrink of the same projection (z = A[l][e] . in, the blog's
// skinny split-K GEMM, section "Kernel optimizations") runs in the same launch
// as "shrink items" ahead of the GEMM tasks: an item stacks the A matrices of
// G = 128 / r consecutive (expert, adapter) buckets on M (slot s = rows
// s*r .. s*r+r-1) against those buckets' pairs -- a contiguous run of rows in
// bucket order -- on N, and each pair keeps its own slot's r rows (the cross
// terms cost tensor time only).  K is split across items when the buckets are
// few; the split that arrives last adds the partials in split order
// (deterministic).  Every shrink item is taken before any GEMM task, and a
// GEMM epilogue reads z only after a device counter shows every shrink task
// finished, so the shrink hides under the weight streaming instead of being a
// launch of its own.
//
// Warp roles (one CTA per SM, persistent; items taken in order from a device
// counter by the producer, which passes each index to the other roles):
//   warp 0   TMA producer: per 64-wide K step, the weight tile (gate_up: the
//            128 gate rows and the 128 matching up rows) and the pairs' rows
//            (x or act in bucket order, 16-row boxes), all 128-byte swizzled,
//            into a ring of shared-memory stages (full/empty mbarriers);
//   warp 1   allocates TMEM; one thread issues tcgen05.mma (M=128, N=n_cols,
//            K=16) into one of two TMEM accumulators (gate_up: a gate and an
//            up accumulator, so a unit's gate and up values land in the same
//            TMEM lane), and commits stage releases and accumulator
//            completion to mbarriers;
//   warps 2-9 epilogue: each thread owns one weight row (its TMEM lane; two
//            warps per lane quadrant take alternate 16-column chunks), adds the
//            LoRA expand B[l][e][row] . z[pair] on CUDA cores when the tensor
//            cores do not take it, and writes bf16 SiLU(gate)*up or bf16 w * d
//            (down with split K: fp32, one slab per split, added by the
//            reduce).  Per task the column metadata (pair,
//            adapter, weight) and the chunk's z rows are first staged in
//            shared memory, while the task's MMAs are still running.
// The two accumulators alternate, so one task's epilogue overlaps the next
// task's MMAs.  Every wait is bounded (tma.cuh); on a timeout the CTA records
// kStatusTimeout, drains its copies, frees TMEM and exits.
#include "gemm_tasks.cuh"

namespace moelora {

namespace {

// depth of the queue that hands the producer's task indices to the MMA and
// epilogue roles
constexpr int kTaskQ = 8;

template <bool GATE_UP, int BN>
struct TcShape {
    static constexpr int kAB = GATE_UP ? 2 * kATile : kATile;  // weight bytes per stage
    static constexpr int kStage = kAB + BN * kBK * 2;          // + pair rows
    static constexpr int kAccCols = GATE_UP ? 2 * BN : BN;      // TMEM columns per accumulator set
    // accumulator sets in TMEM: as many as fit, up to 4, so the MMAs can run
    // ahead of the epilogue on short tasks
    static constexpr int kNAcc = 4 * kAccCols <= 512 ? 4 : 2;
    static constexpr int kTmemCols = kNAcc * kAccCols <= 32 ? 32 : kNAcc * kAccCols;
    static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "TMEM allocation");
    static_assert(BN % 16 == 0 && BN <= 256, "MMA N");
};

// Epilogue state of one thread = one weight row of the tile: the row's LoRA B
// (gate and up rows for gate_up) for the adapter of the current run of pairs.
template <bool GATE_UP>
struct EpiRow {
    int e, w_row, cur_l;
    bool row_ok;
    size_t rows_per_expert;
    float* pout;         // down: this K-split's [P][H] fp32 slab, or
    uint16_t* pout16;    // the [P][H] bf16 output when K is not split
    uint4 bg[8], bu[8];  // r <= 64 bf16 each

    __device__ void init(const TcArgs& a, int e_, int w_row_, bool row_ok_, size_t rpe, float* pout_,
                         uint16_t* pout16_) {
        e = e_;
        w_row = w_row_;
        row_ok = row_ok_;
        rows_per_expert = rpe;
        pout = pout_;
        pout16 = pout16_;
        cur_l = -2;
    }

    // this row of B[l][e] (and its up row for gate_up) for adapter l: runs once
    // per adapter run
    __device__ __forceinline__ void reload(const TcArgs& a, int l) {
        const int r = a.r;
        const size_t gbase = (((size_t)l * a.E + e) * rows_per_expert + w_row) * r;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            if (i * 8 < r) {
                bg[i] = ld_ro16(a.B + gbase + i * 8);
                if (GATE_UP) bu[i] = ld_ro16(a.B + gbase + (size_t)a.I * r + i * 8);
            }
        }
        cur_l = l;
    }

    // one pair of this row (compact row q, pair id p, adapter l, top-k weight
    // w, its z at zq): add the expand, apply the epilogue, store
    __device__ __forceinline__ void column(const TcArgs& a, int q, int p, int l, float w, const float* zq, float vg,
                                           float vu, bool has_lora) {
        const int r = a.r;
        if (has_lora && l >= 0 && row_ok) {
            if (l != cur_l) reload(a, l);  // pairs come grouped by adapter: once per run
            float dg0 = 0.f, dg1 = 0.f, du0 = 0.f, du1 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                if (i * 8 < r) {
                    float zz[8];
                    const float4 z0 = *reinterpret_cast<const float4*>(zq + i * 8);
                    const float4 z1 = *reinterpret_cast<const float4*>(zq + i * 8 + 4);
                    zz[0] = z0.x; zz[1] = z0.y; zz[2] = z0.z; zz[3] = z0.w;
                    zz[4] = z1.x; zz[5] = z1.y; zz[6] = z1.z; zz[7] = z1.w;
                    if (i & 1) dg1 = dot8(bg[i], zz, dg1);
                    else dg0 = dot8(bg[i], zz, dg0);
                    if (GATE_UP) {
                        if (i & 1) du1 = dot8(bu[i], zz, du1);
                        else du0 = dot8(bu[i], zz, du0);
                    }
                }
            }
            vg += dg0 + dg1;
            vu += du0 + du1;
        }
        if (row_ok) {
            if (GATE_UP)
                a.act_out[(size_t)q * a.I + w_row] = f32_to_bf16_rne(silu_f(vg) * vu);
            else if (pout16)
                pout16[(size_t)p * a.H + w_row] = f32_to_bf16_cvt(w * vg);
            else
                pout[(size_t)p * a.H + w_row] = w * vg;
        }
    }
};

template <bool GATE_UP, int BN>
__global__ void __launch_bounds__(kTcThreads, 1) k_moe_gemm_tc(const __grid_constant__ TcArgs a) {
    using S = TcShape<GATE_UP, BN>;
    constexpr int kRows = kRowsFor<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int NS = a.nstages;
    // epilogue staging: z rows [BN][r] fp32, then pair id / adapter / weight per
    // column (a shrink item keeps its slots' column ranges in s_pair / s_lora)
    float* zs = reinterpret_cast<float*>(base + (size_t)NS * S::kStage);
    int* s_pair = reinterpret_cast<int*>(zs + (a.tc_expand ? 0 : (size_t)BN * a.r));
    int* s_lora = s_pair + BN;
    float* s_w = reinterpret_cast<float*>(s_lora + BN);
    int* s_misc = reinterpret_cast<int*>(s_w + BN);  // [kMisc] shared by the epilogue warps
    uint64_t* full = reinterpret_cast<uint64_t*>(s_misc + kMisc);
    uint64_t* empty = full + NS;
    uint64_t* tfull = empty + NS;       // [kNAcc] accumulator ready for the epilogue
    uint64_t* tempty = tfull + S::kNAcc;  // [kNAcc] accumulator drained by the epilogue
    uint64_t* ebar = tempty + S::kNAcc;   // epilogue rendezvous (kEpiWarps * 32 arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ebar + 1);
    uint64_t* tq_full = reinterpret_cast<uint64_t*>(tmem_slot + 4);  // [kTaskQ] task index written
    uint64_t* tq_empty = tq_full + kTaskQ;                            // [kTaskQ] read by the MMA thread and every epilogue warp
    int* tq = reinterpret_cast<int*>(tq_empty + kTaskQ);              // [kTaskQ] task indices
    TaskTable tt;
    tt.cmask = reinterpret_cast<unsigned long long*>(tq + kTaskQ);
    tt.e = reinterpret_cast<int*>(tt.cmask + (a.chunk_masks ? a.max_chunks : 0));
    tt.q0 = tt.e + a.E;
    tt.m = tt.q0 + a.E;
    tt.cum = tt.m + a.E;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < S::kNAcc; b++) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(ebar, kEpiWarps * 32);
        for (int q = 0; q < kTaskQ; q++) {
            mbar_init(&tq_full[q], 1);
            mbar_init(&tq_empty[q], 1 + kEpiWarps);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, S::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&a.wmap);
        prefetch_tensormap(&a.xmap);
        if (a.sh_tasks) prefetch_tensormap(&a.amap);
        if (a.tc_expand) {
            prefetch_tensormap(&a.bmap);
            prefetch_tensormap(&a.bmap1);
            prefetch_tensormap(&a.zxmap);
            prefetch_tensormap(&a.zxmap1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    pdl_wait();
    pdl_trigger();

    const int N_out = GATE_UP ? a.I : a.H;
    const int K = GATE_UP ? a.H : a.I;
    const int ntiles = (N_out + kBM - 1) / kBM;
    const int nkb = (K + kBK - 1) / kBK;
    const int n_active = a.hdr->n_active;
    build_task_table<BN>(a, tt, n_active, ntiles);
    const int ksplit = a.ksplit;
    // shrink items first, then the GEMM tasks
    const bool shrink = a.sh_tasks != nullptr && a.r > 0;
    const bool expand = a.tc_expand != 0 && a.r > 0;
    const int sh_ks = a.sh_ks;
    const int n_sh_tasks = shrink ? a.hdr->n_shrink_tasks : 0;
    const int n_sh = n_sh_tasks * sh_ks;
    const int n_lora = shrink ? a.hdr->n_lora_buckets : 0;
    const int L1 = a.L + 1;
    const int total = n_sh + tt.cum[n_active] * ksplit;
    // Tasks are taken in order: with a task counter each CTA's producer takes
    // the next index when it is ready for a new task (so CTAs that drew cheap
    // tasks take more) and passes it to the MMA thread and the epilogue
    // through the tq queue; without one they are dealt round-robin.  Either
    // way the pair chunks of one weight tile (and the tiles of one expert)
    // stream on neighbouring CTAs at about the same time and share their
    // operands through L2, and every shrink item is taken before any GEMM task.
    const int t_first = blockIdx.x, t_step = gridDim.x;
    const bool dyn = a.task_counter != nullptr;
    // the consumers' view of task it: from the queue, or from the deal
    auto take_task = [&](int it, bool& good) -> int {
        if (!dyn) return t_first + it * t_step;
        const int q = it % kTaskQ;
        good = __all_sync(__activemask(), mbar_wait(&tq_full[q], (uint32_t)(it / kTaskQ) & 1u));
        const int t = good ? tq[q] : total;
        __syncwarp(__activemask());
        // one arrival from the MMA thread and one per epilogue warp
        if (good && (warp == 1 || lane == 0)) mbar_arrive(&tq_empty[q]);
        return t;
    };
    bool ok = true;

    if (warp == 0) {
        // -------------------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, armed = 0, last_par = 0;
            bool z_seen = false;
            int arow[kMaxSlots];
            int t = t_first;
            for (int it = 0; ok; it++) {
                if (dyn) {
                    const int q = it % kTaskQ;
                    if (!mbar_wait(&tq_empty[q], ((uint32_t)(it / kTaskQ) & 1u) ^ 1u)) { ok = false; break; }
                    t = atomicAdd(a.task_counter, 1);
                    tq[q] = t;
                    mbar_arrive(&tq_full[q]);  // also for the end marker t >= total
                } else if (it > 0) {
                    t += t_step;
                }
                if (t >= total) break;
                if (t < n_sh) {
                    // shrink item: one r-row box per slot, then the pair rows
                    ShItem sh;
                    sh.load(a, t, n_lora);
                    for (int q = 0; q < sh.nb; q++) {
                        const int b = a.lora_buckets[sh.j0 + q];
                        arow[q] = ((b % L1 - 1) * a.E + b / L1) * a.r;  // first row of A[l][e]
                    }
                    const int sh_box = (sh.n_cols + kRows - 1) / kRows;
                    const uint32_t bytes = (uint32_t)(sh.nb * a.r + sh_box * kRows) * kBK * 2;
                    const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
                        mbar_arrive_expect_tx(&full[stage], bytes);
                        uint8_t* dst = base + (size_t)stage * S::kStage;
                        const int k0 = kb * kBK;
                        for (int q = 0; q < sh.nb; q++)
                            tma_load_2d(dst + q * a.r * kBK * 2, &a.amap, &full[stage], k0, arow[q]);
                        for (int g = 0; g < sh_box; g++)
                            tma_load_2d(dst + kATile + g * kRows * kBK * 2, &a.xmap, &full[stage], k0, sh.q0c + g * kRows);
                        armed |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                    }
                    continue;
                }
                Task<BN> tw;
                tw.lookup(tt, n_active, ksplit, ntiles, t - n_sh);
                const int n_cols = tw.n_cols, row0 = tw.q0c, e = tw.e;
                const int n_box = (n_cols + kRows - 1) / kRows;
                const uint32_t bytes = S::kAB + (uint32_t)n_box * kRows * kBK * 2;
                const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
                // LoRA expand K-blocks of this task's split (without chunk masks the
                // pair ids are fetched now, their adapters before the last base stage)
                ExpandRange xr;
                xr.none();
                int n_x = 0;
                if (expand && a.chunk_masks) {
                    xr.from_mask(a, tt.cmask[tw.chunk], tw.split, ksplit);
                    n_x = xr.count();
                } else if (expand) {
                    xr.begin(a, row0, tw.n_real);
                }
                for (int kb = kb0; kb < kb1; kb++) {
                    if (expand && !a.chunk_masks && kb == kb1 - 1) {
                        xr.finish_wide(a, tw.split, ksplit);
                        n_x = xr.count();
                    }
                    if (!mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    uint8_t* dst = base + (size_t)stage * S::kStage;
                    const int k0 = kb * kBK;
                    if (GATE_UP) {
                        tma_load_4d(dst, &a.wmap, &full[stage], k0, tw.mt * kBM, 0, e);
                        tma_load_4d(dst + kATile, &a.wmap, &full[stage], k0, tw.mt * kBM, 1, e);
                    } else {
                        tma_load_3d(dst, &a.wmap, &full[stage], k0, tw.mt * kBM, e);
                    }
                    for (int g = 0; g < n_box; g++)
                        tma_load_2d(dst + S::kAB + g * kRows * kBK * 2, &a.xmap, &full[stage], k0, row0 + g * kRows);
                    armed |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
                // the expand reads zexp: wait once until every shrink task is done
                if (ok && n_x > 0 && !z_seen) {
                    if (!wait_count(a.zdone, n_sh_tasks)) { ok = false; break; }
                    // the shrink items' generic stores before the TMA (async proxy) reads
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    z_seen = true;
                }
                // a block's adapters: A sub-tiles (128 x r_pad each, one copy per
                // half) and zexp sub-tiles (BN rows x r_pad each)
                const uint32_t xa1 = 128u * expand_rpad(a.r) * 2u;  // one adapter's A sub-tile
                const uint32_t zx1 = (uint32_t)BN * expand_rpad(a.r) * 2u;  // one adapter's zexp sub-tile
                if (n_x > 0 && !xr.wide) {
                    // packed blocks: the next 64 / r_pad present adapters, one
                    // single-adapter copy each for A (per half) and for zexp
                    // (other splits' groups are skipped by clearing their bits:
                    // this one thread issues every copy of the CTA)
                    unsigned long long rem = xr.bits;
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
                        if (!mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
                        mbar_arrive_expect_tx(&full[stage], (uint32_t)cnt * ((GATE_UP ? 2u : 1u) * xa1 + zx1));
                        uint8_t* dst = base + (size_t)stage * S::kStage;
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            if (q < cnt) {
                                // coordinates (k, unit, half, expert, adapter) / (k, row, expert, adapter)
                                if (GATE_UP) {
                                    tma_load_5d(dst + q * xa1, &a.bmap1, &full[stage], 0, tw.mt * kBM, 0, e, ids[q]);
                                    tma_load_5d(dst + kATile + q * xa1, &a.bmap1, &full[stage], 0, tw.mt * kBM, 1, e,
                                                ids[q]);
                                } else {
                                    tma_load_4d(dst + q * xa1, &a.bmap1, &full[stage], 0, tw.mt * kBM, e, ids[q]);
                                }
                                tma_load_3d(dst + S::kAB + q * zx1, &a.zxmap1, &full[stage], 0, row0, ids[q]);
                            }
                        }
                        armed |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                    }
                }
                for (int jb = (n_x > 0 && xr.wide) ? xr.next(0) : -1; ok && jb >= 0; jb = xr.next(jb + 1)) {
                    // a block with one adapter present loads that adapter's rows only
                    const uint32_t sm = xr.slots(jb);
                    const bool one = __popc(sm) == 1;
                    const uint32_t abytes = one ? xa1 : (uint32_t)kATile;
                    if (!mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], (GATE_UP ? 2u : 1u) * abytes + (uint32_t)BN * kBK * 2u);
                    uint8_t* dst = base + (size_t)stage * S::kStage;
                    const int l0 = jb * xr.apb;
                    const int q1 = __ffs(sm) - 1;
                    const CUtensorMap* bm = one ? &a.bmap1 : &a.bmap;
                    const int la = one ? l0 + q1 : l0;
                    const uint32_t ao = one ? q1 * xa1 : 0u;
                    // coordinates (k, unit, half, expert, adapter) / (k, row, expert, adapter)
                    if (GATE_UP) {
                        tma_load_5d(dst + ao, bm, &full[stage], 0, tw.mt * kBM, 0, e, la);
                        tma_load_5d(dst + kATile + ao, bm, &full[stage], 0, tw.mt * kBM, 1, e, la);
                    } else {
                        tma_load_4d(dst + ao, bm, &full[stage], 0, tw.mt * kBM, e, la);
                    }
                    tma_load_3d(dst + S::kAB, &a.zxmap, &full[stage], 0, row0, l0);
                    armed |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
            }
            // every issued copy lands before the CTA may exit
            for (int s = 0; s < NS; s++)
                if ((armed >> s) & 1u) mbar_wait(&full[s], (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA issuer
        // Walks the same item sequence as the producer (shrink items, then GEMM
        // tasks with their expand K-blocks); task data comes from the shared
        // table.  Descriptors are built by adds from two base descriptors (the
        // start-address field counts 16-byte units: a stage adds kStage / 16, a
        // sub-tile its offset / 16, a 16-wide K step 2), since this one thread
        // issues every MMA of the CTA.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            // expand sub-tiles: r_pad-wide K-major rows, swizzle span = one row
            const int xrp = expand_rpad(a.r);
            const uint32_t xa16 = 128u * xrp * 2u / 16u;  // one adapter's A sub-tile, in 16-byte units
            const uint64_t d0 = umma_desc_sw128(smem_u32(base));
            const uint64_t dx0 = umma_desc_kmajor(smem_u32(base), expand_layout(xrp), 8u * xrp * 2u);
            constexpr uint64_t kStage16 = S::kStage / 16, kUp16 = kATile / 16, kPair16 = S::kAB / 16;
            for (int it = 0; ok; it++) {
                bool good = true;
                const int t = take_task(it, good);
                if (!good) { ok = false; break; }
                if (t >= total) break;
                const int b = it % S::kNAcc;
                if (!mbar_wait(&tempty[b], ((uint32_t)(it / S::kNAcc) & 1u) ^ 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_first = tmem_base + (uint32_t)(b * S::kAccCols);
                if (t < n_sh) {
                    ShItem sh;
                    sh.load(a, t, n_lora);
                    const uint32_t idesc = umma_idesc_bf16_f32(kBM, sh.n_cols);
                    const int kb0 = sh.sp * nkb / sh_ks, kb1 = (sh.sp + 1) * nkb / sh_ks;
                    for (int kb = kb0; kb < kb1; kb++) {
                        if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t da = d0 + (uint64_t)stage * kStage16;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; kk++)
                            umma_bf16(d_first, da + 2 * kk, da + kUp16 + 2 * kk, idesc, (kb != kb0) || (kk != 0));
                        umma_commit(&empty[stage]);
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    umma_commit(&tfull[b]);
                    continue;
                }
                Task<BN> tw;
                tw.lookup(tt, n_active, ksplit, ntiles, t - n_sh);
                const uint32_t idesc = umma_idesc_bf16_f32(kBM, tw.n_cols);
                const int kb0 = tw.split * nkb / ksplit, kb1 = (tw.split + 1) * nkb / ksplit;
                ExpandRange xr;
                xr.none();
                if (expand && a.chunk_masks) {
                    xr.from_mask(a, tt.cmask[tw.chunk], tw.split, ksplit);
                } else if (expand) {
                    // the expand blocks (same rule as the producer), looked up while
                    // the first stage is in flight
                    xr.begin(a, tw.q0c, tw.n_real);
                    xr.finish_wide(a, tw.split, ksplit);
                }
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t da = d0 + (uint64_t)stage * kStage16;
                    const uint64_t db = da + kPair16;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; kk++) {
                        const uint32_t acc = (kb != kb0) || (kk != 0);
                        umma_bf16(d_first, da + 2 * kk, db + 2 * kk, idesc, acc);
                        if (GATE_UP) umma_bf16(d_first + BN, da + kUp16 + 2 * kk, db + 2 * kk, idesc, acc);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
                if (!xr.wide) {
                    // packed blocks of this split: sub-tiles 0 .. cnt-1
                    const int ng = xr.groups();
                    for (int g = xr.split; g < ng && ok; g += xr.ksplit) {
                        const int cnt = xr.group_size(g);
                        if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dxs = dx0 + (uint64_t)stage * kStage16;
                        for (int q = 0; q < cnt; q++) {
                            const uint64_t da = dxs + q * xa16;
                            const uint64_t db = dxs + kPair16 + q * (uint32_t)(BN * xrp * 2 / 16);
                            for (int kk = 0; kk < xrp / 16; kk++) {
                                umma_bf16(d_first, da + 2 * kk, db + 2 * kk, idesc, 1u);
                                if (GATE_UP) umma_bf16(d_first + BN, da + kUp16 + 2 * kk, db + 2 * kk, idesc, 1u);
                            }
                        }
                        umma_commit(&empty[stage]);
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                    }
                }
                for (int jb = xr.wide ? xr.next(0) : -1; jb >= 0 && ok; jb = xr.next(jb + 1)) {
                    const uint32_t sm = xr.slots(jb);
                    if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dxs = dx0 + (uint64_t)stage * kStage16;
                    for (int q = 0; q < xr.apb; q++) {
                        if (!((sm >> q) & 1u)) continue;
                        const uint64_t da = dxs + q * xa16;
                        const uint64_t db = dxs + kPair16 + q * (uint32_t)(BN * xrp * 2 / 16);
                        for (int kk = 0; kk < xrp / 16; kk++) {
                            umma_bf16(d_first, da + 2 * kk, db + 2 * kk, idesc, 1u);
                            if (GATE_UP) umma_bf16(d_first + BN, da + kUp16 + 2 * kk, db + 2 * kk, idesc, 1u);
                        }
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                umma_commit(&tfull[b]);
            }
        }
    } else {
        // -------------------------------------------------------------- epilogue
        const int ew = warp - 2;                 // 0 .. kEpiWarps-1
        const int qd = warp & 3;                 // TMEM lane quadrant of this warp
        const int half = ew >> 2;                // which alternate 16-column chunks
        const int row = qd * 32 + lane;          // weight row within the tile
        const int etid = ew * 32 + lane;
        // the CUDA-core expand runs here only when the tensor cores do not take it
        const bool has_lora = a.B != nullptr && a.z != nullptr && !a.tc_expand;
        const size_t rows_per_expert = GATE_UP ? 2 * (size_t)a.I : (size_t)a.H;
        const int r = a.r;
        uint32_t epar = 0;
        bool z_ready = !has_lora;
        // all epilogue warps meet here (bounded); false on timeout, warp-uniform
        auto rendezvous = [&]() {
            mbar_arrive(ebar);
            const bool r_ok = __all_sync(kFull, mbar_wait(ebar, epar));
            epar ^= 1;
            return r_ok;
        };
        for (int it = 0; ok; it++) {
            bool good = true;
            const int t = take_task(it, good);
            if (!good) { ok = false; break; }
            if (t >= total) break;
            const int b = it % S::kNAcc;
            const int use = it / S::kNAcc;  // how often this accumulator set was used before
            if (t < n_sh) {
                auto release = [&](int bb) { mbar_arrive(&tempty[bb]); };
                if (!shrink_epilogue(a, t, n_lora, b, use, tmem_base, S::kAccCols, qd, half, lane, etid, s_pair,
                                     s_lora, s_misc, tfull, rendezvous, release, 0, 1)) { ok = false; break; }
                continue;
            }
            Task<BN> tw;
            tw.lookup(tt, n_active, ksplit, ntiles, t - n_sh);
            const int e = tw.e, q0c = tw.q0c, n_real = tw.n_real, n_cols = tw.n_cols;
            // z is complete once every shrink task has finished (all are taken before any GEMM task)
            if (!z_ready && etid == 0) s_misc[0] = wait_count(a.zdone, n_sh_tasks);
            // stage this task's column data while its MMAs run (after everyone
            // is done with the previous task's)
            if (!rendezvous()) { ok = false; break; }
            if (!z_ready) {
                if (!s_misc[0]) { ok = false; break; }
                __threadfence();
                z_ready = true;
            }
            for (int c = etid; c < n_real; c += kEpiWarps * 32) {
                const int p = a.compact_ids[q0c + c];
                s_pair[c] = p;
                s_lora[c] = a.lora_ids[p / a.k];
                s_w[c] = a.topk_weights[p];
            }
            if (has_lora) {
                const float4* zsrc = reinterpret_cast<const float4*>(a.z + (size_t)q0c * r);
                float4* zdst = reinterpret_cast<float4*>(zs);
                for (int i = etid; i < n_real * r / 4; i += kEpiWarps * 32) zdst[i] = __ldcg(zsrc + i);
            }
            if (!rendezvous()) { ok = false; break; }

            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(kFull, mbar_wait(&tfull[b], (uint32_t)use & 1u))) { ok = false; break; }
            tc_fence_after();
            const int w_row = tw.mt * kBM + row;
            const bool row_ok = w_row < N_out;
            const uint32_t t_lane = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(b * S::kAccCols);
            // split-K of gate_up: partial tiles go to global memory; the split
            // that arrives last adds the others' partials (in split order) to
            // its own.  Split-K of down: every split writes w * its partial to
            // its own fp32 slab of pair_out (the reduce kernel adds the slabs in
            // split order), so no split waits for another; without a split,
            // w * d goes out in bf16.
            const bool slab = !GATE_UP && ksplit > 1;
            float* const pout = GATE_UP || !slab ? nullptr : a.pair_out + (size_t)tw.split * a.pair_split;
            uint16_t* const pout16 = GATE_UP || slab ? nullptr : a.pair_out16;
            bool finish = true;
            float* part_tile = nullptr;
            if (ksplit > 1 && !slab) {
                part_tile = a.part + (size_t)tw.tile * ksplit * S::kAccCols * kBM;
                float* mine = part_tile + (size_t)tw.split * S::kAccCols * kBM;
                for (int c0 = half * 16; c0 < n_cols; c0 += 32) {
                    float g[16];
                    tmem_ld16(t_lane + c0, g);
#pragma unroll
                    for (int c = 0; c < 16; c++) mine[(size_t)(c0 + c) * kBM + row] = g[c];
                    if (GATE_UP) {
                        tmem_ld16(t_lane + BN + c0, g);
#pragma unroll
                        for (int c = 0; c < 16; c++) mine[(size_t)(BN + c0 + c) * kBM + row] = g[c];
                    }
                }
                __threadfence();
                if (!rendezvous()) { ok = false; break; }
                if (etid == 0) s_misc[1] = atomicAdd(&a.tile_counters[tw.tile], 1) == ksplit - 1;
                if (!rendezvous()) { ok = false; break; }
                finish = s_misc[1] != 0;
                if (finish) __threadfence();
            }
            if (!has_lora && (ksplit == 1 || slab)) {
                // lean epilogue (no CUDA-core expand, no split-K finish): 16
                // columns of each accumulator per TMEM load, one wait for both
                for (int c0 = half * 16; c0 < n_real; c0 += 32) {
                    float g[16], u[16];
                    if (GATE_UP) tmem_ld16x2(t_lane + c0, t_lane + BN + c0, g, u);
                    else tmem_ld16(t_lane + c0, g);
                    if (row_ok) {
#pragma unroll
                        for (int c = 0; c < 16; c++) {
                            const int cc = c0 + c;
                            if (cc < n_real) {
                                if (GATE_UP)
                                    a.act_out[(size_t)(q0c + cc) * a.I + w_row] = f32_to_bf16_cvt(silu_fast(g[c]) * u[c]);
                                else if (!slab)
                                    pout16[(size_t)s_pair[cc] * a.H + w_row] = f32_to_bf16_cvt(s_w[cc] * g[c]);
                                else
                                    pout[(size_t)s_pair[cc] * a.H + w_row] = s_w[cc] * g[c];
                            }
                        }
                    }
                }
                finish = false;
            }
            EpiRow<GATE_UP> er;
            er.init(a, e, w_row, row_ok, rows_per_expert, pout, pout16);
            // the CUDA-core expand is added once: by split 0 when splits write slabs
            const bool add_lora = has_lora && (!slab || tw.split == 0);
            for (int c0 = half * 16; finish && c0 < n_cols; c0 += 32) {
                // columns in groups of four keep the loop small (instruction cache)
                for (int c4 = c0; c4 < c0 + 16 && c4 < n_real; c4 += 4) {
                    float g4[4], u4[4];
                    if (ksplit == 1 || slab) {
                        tmem_ld4(t_lane + c4, g4);
                        if (GATE_UP) tmem_ld4(t_lane + BN + c4, u4);
                    } else {
                        // every split's partial added in split order: this split's own
                        // from TMEM, the others' from global memory, all of a column
                        // group's loads issued before the first add
                        float og[4], ou[4];
                        tmem_ld4(t_lane + c4, og);
                        if (GATE_UP) tmem_ld4(t_lane + BN + c4, ou);
#pragma unroll
                        for (int c = 0; c < 4; c++) g4[c] = u4[c] = 0.f;
                        constexpr int kCols = GATE_UP ? 2 : 4;  // columns per batch of loads
#pragma unroll
                        for (int cb = 0; cb < 4; cb += kCols) {
                            float pg[kMaxKsplit][kCols], pu[kMaxKsplit][kCols];
#pragma unroll
                            for (int sp = 0; sp < kMaxKsplit; sp++) {
                                if (sp < ksplit && sp != tw.split) {
                                    const float* ps = part_tile + (size_t)sp * S::kAccCols * kBM + row;
#pragma unroll
                                    for (int c = 0; c < kCols; c++) {
                                        pg[sp][c] = __ldcg(ps + (size_t)(c4 + cb + c) * kBM);
                                        if (GATE_UP) pu[sp][c] = __ldcg(ps + (size_t)(BN + c4 + cb + c) * kBM);
                                    }
                                }
                            }
#pragma unroll
                            for (int sp = 0; sp < kMaxKsplit; sp++) {
                                if (sp < ksplit) {
#pragma unroll
                                    for (int c = 0; c < kCols; c++) {
                                        g4[cb + c] += sp == tw.split ? og[cb + c] : pg[sp][c];
                                        if (GATE_UP) u4[cb + c] += sp == tw.split ? ou[cb + c] : pu[sp][c];
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int cc = c4 + c;
                        if (cc < n_real)
                            er.column(a, q0c + cc, s_pair[cc], s_lora[cc], s_w[cc], zs + cc * r, g4[c],
                                      GATE_UP ? u4[c] : 0.f, add_lora);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }

    if (!ok) atomicOr(&a.hdr->status, kStatusTimeout);
    // all roles done (every wait above is bounded): release TMEM
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, S::kTmemCols);
}

template <bool G, int BN>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(k_moe_gemm_tc<G, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTcSmemLimit);
}

// ---------------------------------------------------------------- gather
// rows of x in bucket (compact) order, the B operand of the gate_up GEMM:
// `wpr` warps per row (few rows: several warps share one), each row's token
// id read once per warp, lanes over the row's 16-byte chunks
__global__ void __launch_bounds__(256) k_gather_rows(GatherArgs a) {
    pdl_wait();
    pdl_trigger();
    const int n = a.hdr->n_valid;
    const int c8 = a.H >> 3;
    const int lane = threadIdx.x & 31;
    const int wpr = a.wpr;
    const long warps = (long)gridDim.x * (blockDim.x >> 5);
    for (long w = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < (long)n * wpr; w += warps) {
        const int q = (int)(w / wpr), part = (int)(w % wpr);
        const int t = a.compact_ids[q] / a.k;
        const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H);
        uint4* dst = reinterpret_cast<uint4*>(a.out + (size_t)q * a.H);
#pragma unroll 4
        for (int c = part * 32 + lane; c < c8; c += 32 * wpr) dst[c] = ld_ro16(src + c);
    }
    // zexp starts as zeros; the shrink items fill each pair's own adapter
    if (a.zexp1) {
        const long nz = a.zx_elems / 8;
        const long stride = (long)gridDim.x * blockDim.x;
        const uint4 zero = make_uint4(0, 0, 0, 0);
        for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < nz; i += stride) {
            reinterpret_cast<uint4*>(a.zexp1)[i] = zero;
            reinterpret_cast<uint4*>(a.zexp2)[i] = zero;
        }
    }
}

}  // namespace

int tc_smem_bytes(bool gate_up, int bn, int r, int E, int nstages, bool tc_expand, int mask_chunks) {
    const int ab = gate_up ? 2 * kATile : kATile;
    const int stage = ab + bn * kBK * 2;
    const int staging = (tc_expand ? 0 : bn * r * 4) + 3 * bn * 4 + kMisc * 4;
    const int table = 8 * mask_chunks + (4 * E + 1) * 4;
    // at least half an SM's shared memory: one CTA per SM, so a TMEM
    // allocation never waits for another CTA
    const int queue = kTaskQ * (2 * 8 + 4);
    return std::max(1024 + nstages * stage + staging + (2 * nstages + 2 * 4 + 1) * 8 + 16 + queue + table,
                    kTcSmemLimit / 2 + 1024);
}

int tc_plan_stages(bool gate_up, int bn, int r, int E, bool tc_expand, int mask_chunks) {
    for (int ns = 8; ns >= 2; ns--)
        if (tc_smem_bytes(gate_up, bn, r, E, ns, tc_expand, mask_chunks) <= kTcSmemLimit) return ns;
    return 0;
}

cudaError_t init_tc_attributes() {
    cudaError_t e;
    if ((e = set_attr<true, 64>()) != cudaSuccess) return e;
    if ((e = set_attr<true, 128>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 64>()) != cudaSuccess) return e;
    return set_attr<false, 256>();
}

cudaError_t launch_moe_gemm_tc(const TcArgs& args, bool gate_up, int bn, int grid, cudaStream_t stream, bool pdl) {
    const int smem = tc_smem_bytes(gate_up, bn, args.r, args.E, args.nstages, args.tc_expand != 0,
                                   args.chunk_masks ? args.max_chunks : 0);
    const dim3 g(grid), b(kTcThreads);
    if (gate_up) {
        if (bn == 64) return launch_k(k_moe_gemm_tc<true, 64>, g, b, smem, stream, pdl, args);
        return launch_k(k_moe_gemm_tc<true, 128>, g, b, smem, stream, pdl, args);
    }
    if (bn == 64) return launch_k(k_moe_gemm_tc<false, 64>, g, b, smem, stream, pdl, args);
    return launch_k(k_moe_gemm_tc<false, 256>, g, b, smem, stream, pdl, args);
}

cudaError_t launch_gather_rows(const GatherArgs& args, int grid, cudaStream_t stream, bool pdl) {
    return launch_k(k_gather_rows, dim3(grid), dim3(256), 0, stream, pdl, args);
}

}  // namespace moelora
