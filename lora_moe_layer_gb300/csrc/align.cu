// align.cu -- expert x adapter bucketing of the (token, slot) pairs.
//
// The blog ("Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Implementing multi-LoRA
// inference for MoE models in vLLM") describes its fused_moe_lora kernel as
// fused_moe plus one more grid dimension over the active adapters, because
// MoE LoRA mixes two sparsities: expert routing and per-request adapter
// choice.  Here that becomes one stable sort of the pairs by the key
// b = e*(L+1) + (l+1): buckets in ascending b, pairs in ascending p inside a
// bucket, each non-empty bucket padded to a multiple of block_m.
//
// One CTA of 16 warps.  First every thread computes bucket keys for a strided
// share of the pairs (independent loads, many in flight) into shared memory
// when they fit, else the workspace.  Each warp then owns a contiguous segment
// of pairs and keeps a per-bucket histogram row (shared memory when it fits,
// else the workspace).  Pass 1 counts with warp match-any + popc (one leader
// per distinct key per 32 pairs); the histogram rows are then turned into
// per-warp exclusive prefixes, bucket sizes are scanned (warp shuffles) into
// padded and compact offsets, and pass 2 places every pair at
//     offset[b] + (pairs of b in earlier warps) + (earlier lanes of b in this step).
// Walking each segment in order and the warps in order keeps ascending p.
// The padded outputs (sentinels, per-tile expert and adapter) are written only
// for the standalone entry point; the forward works on the compact order and
// places pairs inside a bucket in any order (shared-memory atomics).
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tma.cuh"

namespace moelora {

namespace {

constexpr int kAlignThreads = 512;
constexpr int kAlignWarps = kAlignThreads / 32;
static_assert(kAlignWarps == kAlignRowsStable, "one histogram row per warp on the stable path");

__device__ __forceinline__ int2 warp_incl_scan2(int2 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, v.x, o);
        const int y = __shfl_up_sync(kFull, v.y, o);
        if (lane >= o) {
            v.x += x;
            v.y += y;
        }
    }
    return v;
}

// Block-wide exclusive scan of an int2 per thread; *total gets the sums.
// sw needs kAlignWarps + 1 entries.  Contains __syncthreads.
__device__ int2 block_excl_scan2(int2 v, int2* total, int2* sw) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int2 inc = warp_incl_scan2(v, lane);
    if (lane == 31) sw[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int2 w = lane < kAlignWarps ? sw[lane] : make_int2(0, 0);
        const int2 wi = warp_incl_scan2(w, lane);
        if (lane < kAlignWarps) sw[lane] = make_int2(wi.x - w.x, wi.y - w.y);
        if (lane == 31) sw[kAlignWarps] = wi;
    }
    __syncthreads();
    const int2 base = sw[warp];
    *total = sw[kAlignWarps];
    const int2 r = make_int2(base.x + inc.x - v.x, base.y + inc.y - v.y);
    __syncthreads();
    return r;
}

// Exclusive scan over n items of (f(i), g(i)) written to out_a / out_b
// (n + 1 entries each, the last being the total).  Items are split into
// contiguous per-thread runs.
template <typename F>
__device__ void block_scan_items(int n, F item, int* out_a, int* out_b, int2* sw) {
    const int per = (n + kAlignThreads - 1) / kAlignThreads;
    const int beg = min(n, (int)threadIdx.x * per);
    const int end = min(n, beg + per);
    int2 local = make_int2(0, 0);
    for (int i = beg; i < end; i++) {
        const int2 v = item(i);
        local.x += v.x;
        local.y += v.y;
    }
    int2 total;
    int2 run = block_excl_scan2(local, &total, sw);
    for (int i = beg; i < end; i++) {
        const int2 v = item(i);
        if (out_a) out_a[i] = run.x;
        if (out_b) out_b[i] = run.y;
        run.x += v.x;
        run.y += v.y;
    }
    if (threadIdx.x == 0) {
        if (out_a) out_a[n] = total.x;
        if (out_b) out_b[n] = total.y;
    }
}

__device__ __forceinline__ int4 add4(int4 a, int4 b) { return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ int4 sub4(int4 a, int4 b) { return make_int4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }

__device__ __forceinline__ int4 warp_incl_scan4(int4 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int4 u;
        u.x = __shfl_up_sync(kFull, v.x, o);
        u.y = __shfl_up_sync(kFull, v.y, o);
        u.z = __shfl_up_sync(kFull, v.z, o);
        u.w = __shfl_up_sync(kFull, v.w, o);
        if (lane >= o) v = add4(v, u);
    }
    return v;
}

// Exclusive scan over n bucket items of four counts each: item(b, sub, e)
// gives them (sub = b % L1 and e = b / L1, kept by increments along each
// thread's contiguous run), and emit(b, e, prefix, item) is called once per
// item in order within the run.  The first kScanCache items of a run are
// evaluated once and kept in registers; longer runs evaluate the rest again
// in the second pass.  Every thread gets the totals.  sw needs kAlignWarps + 1
// entries.  Contains __syncthreads.
constexpr int kScanCache = 8;
template <typename F, typename G>
__device__ int4 block_scan4(int n, int L1, F item, G emit, int4* sw) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (n + kAlignThreads - 1) / kAlignThreads;
    const int beg = min(n, (int)threadIdx.x * per);
    const int end = min(n, beg + per);
    const int sub0 = beg % L1, e0 = beg / L1;
    int4 local = make_int4(0, 0, 0, 0);
    int4 cache[kScanCache];
    int sub = sub0, e = e0;
#pragma unroll
    for (int k = 0; k < kScanCache; k++) {
        if (beg + k < end) {
            cache[k] = item(beg + k, sub, e);
            local = add4(local, cache[k]);
            if (++sub == L1) { sub = 0; e++; }
        }
    }
    for (int i = beg + kScanCache; i < end; i++) {
        local = add4(local, item(i, sub, e));
        if (++sub == L1) { sub = 0; e++; }
    }
    const int4 inc = warp_incl_scan4(local, lane);
    if (lane == 31) sw[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int4 w = lane < kAlignWarps ? sw[lane] : make_int4(0, 0, 0, 0);
        const int4 wi = warp_incl_scan4(w, lane);
        if (lane < kAlignWarps) sw[lane] = sub4(wi, w);
        if (lane == 31) sw[kAlignWarps] = wi;
    }
    __syncthreads();
    int4 run = add4(sw[warp], sub4(inc, local));
    const int4 total = sw[kAlignWarps];
    sub = sub0;
    e = e0;
#pragma unroll
    for (int k = 0; k < kScanCache; k++) {
        if (beg + k < end) {
            emit(beg + k, e, run, cache[k]);
            run = add4(run, cache[k]);
            if (++sub == L1) { sub = 0; e++; }
        }
    }
    for (int i = beg + kScanCache; i < end; i++) {
        const int4 v = item(i, sub, e);
        emit(i, e, run, v);
        run = add4(run, v);
        if (++sub == L1) { sub = 0; e++; }
    }
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kAlignThreads, 1) k_align(AlignArgs a) {
    extern __shared__ __align__(16) int smem_hist[];
    __shared__ int2 sw[kAlignWarps + 1];
    __shared__ int4 sw4[kAlignWarps + 1];
    // The first kernel of a forward is launched without a programmatic
    // dependency, so this wait is a no-op; it stays for standalone use.
    pdl_wait();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = a.T * a.k;
    const int L1 = a.L + 1;
    const int NB = a.E * L1;
    // shared memory: [histogram][bucket tables][pair keys], each part optional
    int* sm = smem_hist;
    int* hist = a.hist_global ? a.hist_global : sm;  // [hist_rows][NB] (+1)
    if (!a.hist_global) sm += a.hist_rows * NB + 1;
    // bucket sizes and padded / compact offsets; later steps read them from here
    int* cnt_t = a.tabs_in_smem ? sm : a.bucket_count;
    int* boff_t = a.tabs_in_smem ? sm + NB : a.bucket_offset;
    int* coff_t = a.tabs_in_smem ? sm + 2 * NB + 1 : a.compact_offset;
    if (a.tabs_in_smem) sm += 3 * NB + 2;
    // bucket key of every pair (-1: left out)
    int* keys = a.keys_in_smem ? sm : a.keys_global;
    WsHeader* hdr = a.hdr;

    // The forward only needs each bucket's pairs together: its per-pair results
    // do not depend on their order inside a bucket, so it counts and places
    // with shared-memory atomics on histogram row 0 (the block's count, then
    // its placement cursor); rows 1.. then hold the adapter-bucket list and
    // the last row the experts that have pairs.  The standalone entry point
    // keeps ascending p inside a bucket: per-warp counts with warp match-any
    // in pass 1 (all rows), ranks in pass 2.
    const bool stable = a.full_outputs != 0;
    const bool lists = a.active_experts != nullptr && !stable;
    int* lbs = hist + NB + 1;                      // copy of the adapter-bucket list (lists only)
    int* e_act = hist + 2 * NB + 1;               // [E] experts with pairs (lists only)

    // The first kKeyBatch pairs of each thread: their ids are loaded into
    // registers before the clearing below and before any key is stored (keys
    // may live in global memory, where the compiler must assume they alias
    // the ids), so the loads overlap one another and the clearing.
    constexpr int kKeyBatch = 8;
    int ev[kKeyBatch], lv[kKeyBatch];
#pragma unroll
    for (int i = 0; i < kKeyBatch; i++) {
        const int p = threadIdx.x + i * kAlignThreads;
        if (p < P) {
            ev[i] = a.topk_ids[p];
            lv[i] = a.lora_ids[p / a.k];
        }
    }
    if (threadIdx.x == 0) hdr->status = 0;
    const int n_hist = stable ? kAlignWarps * NB : NB;
    for (int i = threadIdx.x; i < n_hist; i += kAlignThreads) hist[i] = 0;
    if (lists)
        for (int i = threadIdx.x; i < a.E; i += kAlignThreads) e_act[i] = 0;
    for (int i = threadIdx.x; i < a.n_zero; i += kAlignThreads) a.zero_ints[i] = 0;
    for (int i = threadIdx.x; i < a.n_zero2; i += kAlignThreads) a.zero_ints2[i] = 0;
    int bad = 0;
    {
        auto key = [&](int e, int l) {
            const bool e_ok = e >= 0 && e < a.E;
            const bool l_ok = l >= -1 && l < a.L;
            bad |= (e_ok ? 0 : kStatusBadExpert) | (l_ok ? 0 : kStatusBadLora);
            return e_ok && l_ok ? e * L1 + (l + 1) : -1;
        };
#pragma unroll
        for (int i = 0; i < kKeyBatch; i++) {
            const int p = threadIdx.x + i * kAlignThreads;
            if (p < P) keys[p] = key(ev[i], lv[i]);
        }
        for (int p = threadIdx.x + kKeyBatch * kAlignThreads; p < P; p += kAlignThreads)
            keys[p] = key(a.topk_ids[p], a.lora_ids[p / a.k]);
    }
    __syncthreads();
    // after the barrier, so thread 0's clearing of the status word comes first
    if (bad) atomicOr(&hdr->status, bad);

    // each warp owns pairs [seg_beg, seg_end), walked 32 at a time
    const int seg = ((P + kAlignWarps - 1) / kAlignWarps + 31) & ~31;
    const int seg_beg = min(P, warp * seg);
    const int seg_end = min(P, seg_beg + seg);
    int* my_hist = hist + warp * NB;
    const int run = ((P + kAlignThreads - 1) / kAlignThreads) | 1;  // pairs per thread, odd
    const int run0 = threadIdx.x * run;
    if (stable) {
        // pass 1: per-warp bucket counts
        for (int base = seg_beg; base < seg_end; base += 32) {
            const int p = base + lane;
            const int b = p < seg_end ? keys[p] : -1;
            const unsigned peers = __match_any_sync(kFull, b);
            if (b >= 0 && lane == __ffs(peers) - 1) my_hist[b] += __popc(peers);
            __syncwarp();
        }
    } else {
        // each thread walks its own run of pairs, so one step's atomics spread
        // over the whole batch (consecutive pairs mostly share a bucket); an
        // odd run length keeps the shared-memory key reads free of bank conflicts
#pragma unroll 4
        for (int s = 0; s < run; s++) {
            const int p = run0 + s;
            const int b = p < P ? keys[p] : -1;
            if (b >= 0) {
                atomicAdd(&hist[b], 1);
                if (lists) e_act[b / L1] = 1;
            }
        }
    }
    __syncthreads();

    // per bucket: the bucket size (stable: and the exclusive prefix over warps)
    for (int b = threadIdx.x; b < NB; b += kAlignThreads) {
        int run = 0;
        if (stable) {
            for (int w = 0; w < kAlignWarps; w++) {
                const int c = hist[w * NB + b];
                hist[w * NB + b] = run;
                run += c;
            }
        } else {
            run = hist[b];
            hist[b] = 0;
        }
        cnt_t[b] = run;
        // (the forward's kernels read only the compact offsets)
        if (a.tabs_in_smem && !lists) a.bucket_count[b] = run;
    }
    __syncthreads();

    // one scan over the buckets: padded offsets (bucket_offset), compact
    // offsets, and for the forward the list of (e, l >= 0) buckets with pairs
    // and the list of experts with pairs (counted at each expert's first bucket)
    const int bm = a.bm;  // a power of two
    const int* cnt = cnt_t;
    const int4 tot = block_scan4(
        NB, L1,
        [&](int b, int sub, int e) {
            const int c = cnt[b];
            return make_int4((c + bm - 1) & -bm, c, lists && sub != 0 && c > 0 ? 1 : 0,
                             lists && sub == 0 && e_act[e] ? 1 : 0);
        },
        [&](int b, int e, int4 pre, int4 v) {
            boff_t[b] = pre.x;
            coff_t[b] = pre.y;
            if (a.tabs_in_smem) {
                if (!lists) a.bucket_offset[b] = pre.x;
                a.compact_offset[b] = pre.y;
            }
            if (v.z) {
                a.lora_buckets[pre.z] = b;
                lbs[pre.z] = b;
            }
            if (v.w) a.active_experts[pre.w] = e;
        },
        sw4);
    if (threadIdx.x == 0) {
        boff_t[NB] = tot.x;
        coff_t[NB] = tot.y;
        if (a.tabs_in_smem) {
            a.bucket_offset[NB] = tot.x;
            a.compact_offset[NB] = tot.y;
        }
        hdr->num_post_padded = tot.x;
        hdr->n_valid = tot.y;
        if (a.num_post_padded) *a.num_post_padded = tot.x;
        if (lists) {
            hdr->n_lora_buckets = tot.z;
            hdr->n_active = tot.w;
        }
    }
    __syncthreads();

    // pass 2: placement
    if (stable) {
        for (int base = seg_beg; base < seg_end; base += 32) {
            const int p = base + lane;
            const int b = p < seg_end ? keys[p] : -1;
            const unsigned peers = __match_any_sync(kFull, b);
            if (b >= 0) {
                const int rank = my_hist[b] + __popc(peers & lanemask_lt());
                a.sorted_ids[boff_t[b] + rank] = p;
                a.compact_ids[coff_t[b] + rank] = p;
            }
            __syncwarp();
            if (b >= 0 && lane == __ffs(peers) - 1) my_hist[b] += __popc(peers);
            __syncwarp();
        }
    } else {
#pragma unroll 4
        for (int s = 0; s < run; s++) {
            const int p = run0 + s;
            const int b = p < P ? keys[p] : -1;
            if (b >= 0) a.compact_ids[coff_t[b] + atomicAdd(&hist[b], 1)] = p;
        }
    }

    if (a.full_outputs) {
        __syncthreads();
        // padding sentinels, and each bucket's tiles tagged with its (expert, adapter)
        for (int b = threadIdx.x; b < NB; b += kAlignThreads) {
            const int beg = boff_t[b], end = boff_t[b + 1];
            for (int q = beg + cnt[b]; q < end; q++) a.sorted_ids[q] = P;
            for (int q = beg / bm; q < end / bm; q++) {
                a.tile_expert[q] = b / L1;
                a.tile_lora[q] = b % L1 - 1;
            }
        }
    }
    if (lists && a.st_tasks) {
        // shrink tasks: st_G consecutive adapter buckets per group; a group's
        // rows are contiguous in bucket order and split into chunks of st_BN.
        // The scan's output reuses histogram row 0, free after the placement.
        __syncthreads();
        int* tmp = hist;
        const int n = tot.z;
        const int G = a.st_G, BN = a.st_BN;
        const int ng = (n + G - 1) / G;
        const int* coff = coff_t;
        auto rows = [&](int g) {
            const int j1 = min(n, g * G + G) - 1;
            return make_int2(coff[lbs[g * G]], coff[lbs[j1] + 1]);
        };
        block_scan_items(
            ng, [&](int g) { const int2 q = rows(g); return make_int2((q.y - q.x + BN - 1) / BN, 0); },
            tmp, nullptr, sw);
        __syncthreads();
        for (int g = threadIdx.x; g < ng; g += kAlignThreads) {
            const int2 q = rows(g);
            int at = tmp[g];
            for (int q0 = q.x; q0 < q.y; q0 += BN) a.st_tasks[at++] = make_int4(g, q0, min(BN, q.y - q0), 0);
        }
        if (threadIdx.x == 0) hdr->n_shrink_tasks = tmp[ng];
    }
    pdl_trigger();
}

// The forward's align on several CTAs.  Each CTA takes a contiguous slice of
// the pairs: it computes their keys, counts them per bucket in shared memory
// and adds its counts to the global per-bucket counts, whose old values give
// its base inside each bucket.  The CTA that arrives last then sees every
// count: it scans them into the bucket offsets, writes the expert and
// adapter-bucket lists and the shrink task list (as the single-CTA kernel),
// and raises a flag; every CTA waits for the flag (bounded; all CTAs of the
// launch are resident, one per SM) and places its pairs at
//     compact offset of b + its base in b + its own running count of b.
// The counts and sync words start from zero: the forward clears them with a
// memset right before the launch.
__global__ void __launch_bounds__(kAlignThreads, 1) k_align_multi(AlignArgs a) {
    extern __shared__ __align__(16) int sm_multi[];
    __shared__ int2 sw[kAlignWarps + 1];
    __shared__ int4 sw4[kAlignWarps + 1];
    __shared__ int s_last, s_ok;
    pdl_wait();
    const int tid = threadIdx.x;
    const int P = a.T * a.k, L1 = a.L + 1, NB = a.E * L1;
    const int G = gridDim.x, cta = blockIdx.x;
    const int per = (P + G - 1) / G;
    const int p0 = min(P, cta * per), p1 = min(P, p0 + per);
    // shared memory: [NB] counts, [NB] bases, [NB] cursors, [NB + 1] offsets,
    // [NB] adapter-bucket list, [NB] task scan, [per] keys
    int* cnt = sm_multi;
    int* cbase = cnt + NB;
    int* cur = cbase + NB;
    int* coff = cur + NB;
    int* lbs = coff + NB + 1;
    int* tmp = lbs + NB;
    int* keys = tmp + NB;
    WsHeader* hdr = a.hdr;

    for (int i = tid; i < NB; i += kAlignThreads) {
        cnt[i] = 0;
        cur[i] = 0;
    }
    // the counters of the kernels that follow (grid-stride over all CTAs)
    for (int i = cta * kAlignThreads + tid; i < a.n_zero; i += G * kAlignThreads) a.zero_ints[i] = 0;
    for (int i = cta * kAlignThreads + tid; i < a.n_zero2; i += G * kAlignThreads) a.zero_ints2[i] = 0;
    __syncthreads();
    {
        int bad = 0;
#pragma unroll 4
        for (int p = p0 + tid; p < p1; p += kAlignThreads) {
            const int e = a.topk_ids[p];
            const int l = a.lora_ids[p / a.k];
            const bool e_ok = e >= 0 && e < a.E;
            const bool l_ok = l >= -1 && l < a.L;
            const int b = e_ok && l_ok ? e * L1 + (l + 1) : -1;
            keys[p - p0] = b;
            if (b >= 0) atomicAdd(&cnt[b], 1);
            bad |= (e_ok ? 0 : kStatusBadExpert) | (l_ok ? 0 : kStatusBadLora);
        }
        if (bad) atomicOr(&a.sync[2], bad);
    }
    __syncthreads();
    // this CTA's share of each bucket, and where it starts inside the bucket
    for (int b = tid; b < NB; b += kAlignThreads) {
        const int c = cnt[b];
        cbase[b] = c ? atomicAdd(&a.gcount[b], c) : 0;
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&a.sync[0], 1) == G - 1;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int b = tid; b < NB; b += kAlignThreads) cnt[b] = __ldcg(a.gcount + b);
        __syncthreads();
        const int bm = a.bm;  // a power of two
        const int4 tot = block_scan4(
            NB, L1,
            [&](int b, int sub, int) {
                const int c = cnt[b];
                int any = 0;
                if (sub == 0)
                    for (int j = 0; j < L1; j++) any |= cnt[b + j];
                return make_int4((c + bm - 1) & -bm, c, sub != 0 && c > 0 ? 1 : 0, any != 0 ? 1 : 0);
            },
            [&](int b, int e, int4 pre, int4 v) {
                // (the forward's kernels read only the compact offsets)
                a.compact_offset[b] = pre.y;
                coff[b] = pre.y;
                if (v.z) {
                    a.lora_buckets[pre.z] = b;
                    lbs[pre.z] = b;
                }
                if (v.w) a.active_experts[pre.w] = e;
            },
            sw4);
        if (tid == 0) {
            coff[NB] = tot.y;
            a.compact_offset[NB] = tot.y;
            hdr->num_post_padded = tot.x;
            hdr->n_valid = tot.y;
            hdr->n_lora_buckets = tot.z;
            hdr->n_active = tot.w;
            hdr->status = __ldcg(a.sync + 2);
        }
        __syncthreads();
        if (a.st_tasks) {
            // shrink tasks: st_G consecutive adapter buckets per group, each
            // group's rows (contiguous in bucket order) in chunks of st_BN
            const int n = tot.z;
            const int Gs = a.st_G, BN = a.st_BN;
            const int ng = (n + Gs - 1) / Gs;
            auto rows = [&](int g) {
                const int j1 = min(n, g * Gs + Gs) - 1;
                return make_int2(coff[lbs[g * Gs]], coff[lbs[j1] + 1]);
            };
            block_scan_items(
                ng, [&](int g) { const int2 q = rows(g); return make_int2((q.y - q.x + BN - 1) / BN, 0); }, tmp,
                nullptr, sw);
            __syncthreads();
            for (int g = tid; g < ng; g += kAlignThreads) {
                const int2 q = rows(g);
                int at = tmp[g];
                for (int q0 = q.x; q0 < q.y; q0 += BN) a.st_tasks[at++] = make_int4(g, q0, min(BN, q.y - q0), 0);
            }
            if (tid == 0) hdr->n_shrink_tasks = tmp[ng];
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a.sync + 1), "r"(1) : "memory");
        }
    }
    // placement, once the offsets are out
    if (tid == 0) s_ok = wait_count(a.sync + 1, 1);
    __syncthreads();
    if (!s_ok) {
        if (tid == 0) atomicOr(&hdr->status, kStatusTimeout);
        return;
    }
    if (!s_last)
        for (int b = tid; b <= NB; b += kAlignThreads) coff[b] = __ldcg(a.compact_offset + b);
    __syncthreads();
#pragma unroll 4
    for (int p = p0 + tid; p < p1; p += kAlignThreads) {
        const int b = keys[p - p0];
        if (b >= 0) a.compact_ids[coff[b] + cbase[b] + atomicAdd(&cur[b], 1)] = p;
    }
    pdl_trigger();
}

}  // namespace

int align_multi_ctas(long P, int sms) {
    return (int)std::max<long>(1, std::min<long>((P + kAlignThreads - 1) / kAlignThreads, sms));
}

int align_multi_smem_bytes(int E, int L, long P, int ctas) {
    const long nb = (long)E * (L + 1);
    const long per = (P + ctas - 1) / std::max(ctas, 1);
    const long bytes = (6 * nb + 1 + per) * (long)sizeof(int);
    return bytes <= kAlignMaxSmem ? (int)bytes : 0;
}

cudaError_t launch_align_multi(const AlignArgs& args, int ctas, int smem_bytes, cudaStream_t stream) {
    return launch_k(k_align_multi, dim3(ctas), dim3(kAlignThreads), smem_bytes, stream, false, args);
}

// Optional shared-memory parts after the histogram (which must be there too):
// the bucket tables first, then the pair keys, as long as the total fits.
// `rows`: histogram rows of NB ints (kAlignWarps for the standalone entry
// point's per-warp counts, kAlignRowsForward for the forward).
int align_tabs_smem_bytes(int E, int L, int rows) {
    const int hist = align_hist_smem_bytes(E, L, rows);
    const long bytes = (3L * E * (L + 1) + 2) * (long)sizeof(int);
    return hist && hist + bytes <= kAlignMaxSmem ? (int)bytes : 0;
}

int align_keys_smem_bytes(int E, int L, long P, int rows) {
    const long bytes = P * (long)sizeof(int);
    return align_hist_smem_bytes(E, L, rows) + align_tabs_smem_bytes(E, L, rows) + bytes <= kAlignMaxSmem ? (int)bytes
                                                                                                          : 0;
}

int align_smem_bytes(int E, int L, long P, int rows) {
    return align_hist_smem_bytes(E, L, rows) + align_tabs_smem_bytes(E, L, rows) + align_keys_smem_bytes(E, L, P, rows);
}

int align_hist_smem_bytes(int E, int L, int rows) {
    const long nb = (long)E * (L + 1);
    const long bytes = (nb * rows + 1) * (long)sizeof(int);
    return bytes <= kAlignMaxSmemHist ? (int)bytes : 0;
}

long align_hist_global_ints(int E, int L) {
    return align_hist_smem_bytes(E, L, kAlignWarps) ? 0 : (long)E * (L + 1) * kAlignWarps + 1;
}

cudaError_t init_align_attributes() {
    const cudaError_t e = cudaFuncSetAttribute(k_align, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlignMaxSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_align_multi, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlignMaxSmem);
}

cudaError_t launch_align(const AlignArgs& args, int smem_bytes, cudaStream_t stream) {
    // first kernel of a forward: ordinary stream order behind whatever ran before
    return launch_k(k_align, dim3(1), dim3(kAlignThreads), smem_bytes, stream, false, args);
}

}  // namespace moelora
