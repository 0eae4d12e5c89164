// gemm_tasks.cuh -- pieces shared by the two tensor-core GEMM kernels (one
// CTA per weight tile, moe_gemm_tc.cu; a CTA pair per weight tile,
// moe_gemm_2sm.cu): tile constants, the task table and its lookup, the LoRA
// expand block walk, and the LoRA shrink items with their epilogue.
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace moelora {

namespace {

constexpr int kEpiWarps = 8;             // two per TMEM lane quadrant, splitting the columns
constexpr int kTcThreads = (2 + kEpiWarps) * 32;
constexpr int kBM = 128;                 // weight rows per task (MMA M)
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row
constexpr int kATile = kBM * kBK * 2;    // 16 KiB
// pair rows per TMA box: 16 for decode-sized chunks, 64 for 128-pair chunks,
// one 256-row box for 256-pair chunks (fewer, larger copies keep the TMA
// issue rate off the critical path)
template <int BN>
constexpr int kRowsFor = BN >= 256 ? 256 : BN >= 128 ? 64 : 16;
constexpr int kMisc = 36;  // shared verdicts [0..3] and shrink-slot adapters [4..35]
constexpr int kMaxKsplit = 8;  // K-splits of a GEMM task (the host plans at most this many)

__device__ __forceinline__ float silu_f(float u) { return u / (1.0f + expf(-u)); }
// the same with the fast exponential and division intrinsics, for the lean
// epilogue (its result is rounded to bf16)
__device__ __forceinline__ float silu_fast(float u) { return __fdividef(u, 1.0f + __expf(-u)); }

// Task table built once per CTA in shared memory: for active expert a,
// expert id, first pair row, pair count, and the exclusive prefix of its task
// count (weight tiles x pair chunks).  A task index maps to (expert, tile,
// chunk) by a binary search over the prefix.
struct TaskTable {
    unsigned long long* cmask;  // [chunks] adapters (< 64) with pairs in each (expert, pair chunk)
    int* e;    // [n_active]
    int* q0;   // [n_active]
    int* m;    // [n_active]
    int* cum;  // [n_active + 1]
};

template <int BN>
struct Task {
    int ai, e, mt, q0c, n_real, n_cols;
    int chunk;      // (expert, pair chunk) index, for the chunk's adapter mask
    int tile;       // (expert, weight tile, pair chunk) index, for split-K partials
    int split;      // K-split of this task
    __device__ void lookup(const TaskTable& tt, int n_active, int ksplit, int ntiles, int t) {
        tile = t / ksplit;
        split = t % ksplit;
        int lo = 0, hi = n_active;  // last a with cum[a] <= tile
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tt.cum[mid] <= tile) lo = mid;
            else hi = mid;
        }
        ai = lo;
        const int nch = (tt.m[lo] + BN - 1) / BN;
        const int loc = tile - tt.cum[lo];
        mt = loc / nch;
        const int ch = loc % nch;
        chunk = tt.cum[lo] / ntiles + ch;
        e = tt.e[lo];
        q0c = tt.q0[lo] + ch * BN;
        n_real = min(BN, tt.m[lo] - ch * BN);
        n_cols = (n_real + 15) & ~15;
    }
};

// Per-CTA task table in shared memory (every thread of the CTA calls this):
// the active experts' first pair row, pair count and the prefix of their task
// counts (ntiles weight tiles x chunks of BN pairs), then, with chunk masks,
// the adapters present in each (expert, pair chunk).
template <int BN>
__device__ void build_task_table(const TcArgs& a, const TaskTable& tt, int n_active, int ntiles) {
    // task table: independent loads across threads, then one warp scans the counts
    for (int ai = threadIdx.x; ai < n_active; ai += blockDim.x) {
        const int L1 = a.L + 1;
        const int e = a.active_experts[ai];
        const int q0 = a.compact_offset[e * L1];
        const int m = a.compact_offset[(e + 1) * L1] - q0;
        tt.e[ai] = e;
        tt.q0[ai] = q0;
        tt.m[ai] = m;
        tt.cum[ai + 1] = ntiles * ((m + BN - 1) / BN);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < n_active; base += 32) {
            const int i = base + lane;
            int v = i < n_active ? tt.cum[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, v, o);
                if (lane >= o) v += y;
            }
            if (i < n_active) tt.cum[i + 1] = carry + v;
            carry += __shfl_sync(kFull, v, 31);
        }
        if (lane == 0) tt.cum[0] = 0;
    }
    __syncthreads();
    if (a.chunk_masks) {
        // adapters with pairs in each (expert, pair chunk): one item per (expert,
        // adapter) bucket, OR-ed into the chunks the bucket's rows fall in
        const int n_chunks = tt.cum[n_active] / ntiles;
        for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) tt.cmask[c] = 0ull;
        __syncthreads();
        for (int w = threadIdx.x; w < n_active * a.L; w += blockDim.x) {
            const int ai = w / a.L, l = w % a.L;
            const int b = tt.e[ai] * (a.L + 1) + l + 1;
            const int lo = a.compact_offset[b] - tt.q0[ai], hi = a.compact_offset[b + 1] - tt.q0[ai];
            const int c0 = tt.cum[ai] / ntiles;
            for (int ch = lo / BN; hi > lo && ch <= (hi - 1) / BN; ch++) atomicOr(&tt.cmask[c0 + ch], 1ull << l);
        }
        __syncthreads();
    }
}

// LoRA expand on the tensor cores.  An adapter's share of the expand is a
// K-major tile pair of width r_pad (r rounded up to 16, 32 or 64; TMA reads
// zeros beyond r): A = its B rows (128 weight rows x r_pad), B = its zexp rows
// (pairs x r_pad).  zexp [L][P][r_pad] holds, per adapter, every pair's z for
// pairs of that adapter and zeros for all others.  The tiles use the swizzle
// whose span is one row (32, 64 or 128 bytes).  The 64 / r_pad adapters of one
// block share a ring stage as consecutive sub-tiles, loaded by one copy each
// for A (the adapter is the outermost box dimension) and for zexp.
__host__ __device__ inline int expand_rpad(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : 64; }
__device__ inline uint32_t expand_layout(int rp) { return rp == 16 ? 6u : rp == 32 ? 4u : 2u; }

// The expand blocks of one GEMM task.  With up to 64 adapters the chunk's
// adapter set comes from its mask (built at kernel start) and the blocks are
// packed: block g holds the g-th group of 64 / r_pad adapters present in the
// chunk, in id order, each loaded into its own sub-tile.  Beyond 64 adapters,
// the pairs of a chunk (sorted by adapter) span the adapters la .. lb of its
// first and last pair, read from global memory, and block jb covers the fixed
// adapter range jb*apb .. jb*apb+apb-1 of the span (zexp zeros make absent
// adapters add nothing).  Either way, block j goes to the task's K-split
// j mod ksplit, so a split-K task spreads its expand work too (with one
// adapter per block, adapter l goes to split l mod ksplit).
struct ExpandRange {
    int la, lb, p0, p1, split, ksplit, apb, L;
    bool wide;
    unsigned long long bits;   // adapters (ids < 64) present in the chunk
    __device__ void from_mask(const TcArgs& a, unsigned long long m, int split_, int ksplit_) {
        la = 0;
        lb = -1;
        split = split_;
        ksplit = ksplit_;
        apb = 64 / expand_rpad(a.r);
        L = a.L;
        wide = false;
        bits = m;
        if (apb == 1 && ksplit > 1) {
            // one adapter per block: deal the blocks by adapter id, so each
            // split walks only its own adapters
            unsigned long long own = 0ull;
            for (int l = split; l < 64; l += ksplit) own |= 1ull << l;
            bits &= own;
            split = 0;
            ksplit = 1;
        }
    }
    // pair ids of the chunk's first and last row (issued early), then their adapters
    __device__ void begin(const TcArgs& a, int q0c, int n_real) {
        p0 = a.compact_ids[q0c];
        p1 = a.compact_ids[q0c + n_real - 1];
    }
    __device__ void finish_wide(const TcArgs& a, int split_, int ksplit_) {
        la = max(a.lora_ids[p0 / a.k], 0);
        lb = a.lora_ids[p1 / a.k];
        split = split_;
        ksplit = ksplit_;
        apb = 64 / expand_rpad(a.r);
        L = a.L;
        wide = true;
        bits = 0;
    }
    __device__ void none() { la = 0; lb = -1; split = 0; ksplit = 1; apb = 1; L = 0; wide = false; bits = 0; }
    // packed blocks: how many the chunk has, and how many adapters block g holds
    __device__ int groups() const { return (__popcll(bits) + apb - 1) / apb; }
    __device__ int group_size(int g) const { return min(apb, __popcll(bits) - g * apb); }
    // fixed blocks (beyond 64 adapters): first block >= jb of this task's split, or -1
    __device__ int next(int jb) const {
        for (jb = max(jb, la / apb); jb * apb <= lb; jb++)
            if (jb % ksplit == split) return jb;
        return -1;
    }
    // adapters of fixed block jb (bit s = adapter jb*apb + s)
    __device__ uint32_t slots(int jb) const {
        uint32_t sm = 0;
        for (int s = 0; s < apb; s++) {
            const int l = jb * apb + s;
            if (l >= la && l <= lb && l < L) sm |= 1u << s;
        }
        return sm;
    }
    // this split's expand blocks
    __device__ int count() const {
        if (!wide) {
            const int ng = groups();
            return ng > split ? (ng - 1 - split) / ksplit + 1 : 0;
        }
        int n = 0;
        for (int jb = next(0); jb >= 0; jb = next(jb + 1)) n++;
        return n;
    }
};

// ---------------------------------------------------------------- shrink items
constexpr int kMaxSlots = 16;  // adapter buckets per shrink item: 128 / r with r >= 8

// shrink item t: task t / sh_ks of align's list (G buckets from bucket-list
// index j0, pair rows q0c .. q0c + n_real), K-split sp
struct ShItem {
    int i, sp, j0, nb, q0c, n_real, n_cols;
    __device__ void load(const TcArgs& a, int t, int n_lora) {
        i = t / a.sh_ks;
        sp = t % a.sh_ks;
        const int4 v = __ldcg(a.sh_tasks + i);
        j0 = v.x * a.sh_G;
        nb = min(a.sh_G, n_lora - j0);
        q0c = v.y;
        n_real = v.z;
        n_cols = (n_real + 15) & ~15;
    }
};

// Epilogue of shrink item t (in accumulator set b, used `use` times before):
// each thread is one TMEM lane = (slot, rank
// index) row and stores z for the pairs of its slot; the two warps of a lane
// quadrant take alternate 4-column groups.  With a K-split, the split that
// arrives last sums all partials in split order.  The item then counts
// itself in zdone.  False on a timeout (warp-uniform).
//
// With a CTA pair (nranks = 2) an item holds up to 2 * 128 / r buckets: the
// CTA of rank q owns slots q * 128 / r .. (q + 1) * 128 / r - 1 (its TMEM
// lanes), writes those slots' z, counts its own split arrivals, and counts
// itself once in zdone (which then reaches 2 per item).  release(b) frees
// accumulator set b (called by lane 0 of every epilogue warp).
template <typename Rdv, typename Rel>
__device__ bool shrink_epilogue(const TcArgs& a, int t, int n_lora, int b, int use, uint32_t tmem_base,
                                uint32_t acc_cols, int qd, int half, int lane, int etid, int* s_cb, int* s_ce,
                                int* s_misc, uint64_t* tfull, Rdv& rendezvous, Rel& release, int rank,
                                int nranks) {
    ShItem sh;
    sh.load(a, t, n_lora);
    const int r = a.r;
    const int g_cta = 128 / r;               // slots per CTA
    const int g0 = rank * g_cta;             // this CTA's first slot
    const int g1 = min(sh.nb, g0 + g_cta);   // one past its last
    // slot column ranges (after everyone is done with the previous item's staging)
    if (!rendezvous()) return false;
    int* s_sl = s_misc + 4;  // adapter of each slot
    if (etid < sh.nb) {
        const int bk = a.lora_buckets[sh.j0 + etid];
        s_cb[etid] = min(max(a.compact_offset[bk] - sh.q0c, 0), sh.n_real);
        s_ce[etid] = min(max(a.compact_offset[bk + 1] - sh.q0c, 0), sh.n_real);
        s_sl[etid] = bk % (a.L + 1) - 1;
    }
    if (!rendezvous()) return false;
    const int row = qd * 32 + lane;
    const int my_s = g0 + row / r, j = row % r;
    const int s_lo = g0 + (qd * 32) / r, s_hi = min(g0 + (qd * 32 + 31) / r, sh.nb - 1);
    const bool mine = row / r < g_cta && my_s < sh.nb;
    const int mcb = mine ? s_cb[my_s] : 0, mce = mine ? s_ce[my_s] : 0;
    const int clo = s_lo < sh.nb ? s_cb[s_lo] : 0;
    const int chi = s_lo < sh.nb ? s_ce[s_hi] : 0;
    float* dst = a.sh_ks > 1 ? a.zpart + (size_t)sh.sp * a.P * r : a.z;
    // bf16 copy for the tensor-core expand: zexp[l][q][0:r] for the pair in row q
    const int rp = expand_rpad(r);
    uint16_t* zx = (a.zexp != nullptr && a.sh_ks == 1 && mine) ? a.zexp + (size_t)s_sl[my_s] * a.P * rp + j : nullptr;

    if (!__all_sync(kFull, mbar_wait(&tfull[b], (uint32_t)use & 1u))) return false;
    tc_fence_after();
    const uint32_t t_lane = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)b * acc_cols;
    for (int c4 = (clo & ~3) + 4 * half; c4 < chi; c4 += 8) {
        float v[4];
        tmem_ld4(t_lane + c4, v);
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const int cc = c4 + c;
            if (cc >= mcb && cc < mce) {
                dst[(size_t)(sh.q0c + cc) * r + j] = v[c];
                if (zx) zx[(size_t)(sh.q0c + cc) * rp] = f32_to_bf16_rne(v[c]);
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release(b);
    __threadfence();
    if (!rendezvous()) return false;
    if (a.sh_ks > 1) {
        if (etid == 0) s_misc[1] = atomicAdd(&a.sh_counters[sh.i * nranks + rank], 1) == a.sh_ks - 1;
        if (!rendezvous()) return false;
        if (!s_misc[1]) return true;  // the last split of this CTA's part counts it
        if (g1 <= g0) {
            if (etid == 0) atomicAdd(a.zdone, 1);
            return true;
        }
        // one flat pass over the rows this CTA's slots cover (rows of
        // base-only pairs in between get a sum nobody reads)
        __threadfence();
        const int lo = s_cb[g0], hi = s_ce[g1 - 1];
        const size_t beg = (size_t)(sh.q0c + lo) * r;
        const int n4 = (hi - lo) * r / 4;
        const float4* src = reinterpret_cast<const float4*>(a.zpart + beg);
        float4* out = reinterpret_cast<float4*>(a.z + beg);
        const size_t split4 = (size_t)a.P * r / 4;
        for (int i4 = etid; i4 < n4; i4 += kEpiWarps * 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int q = 0; q < a.sh_ks; q++) {
                const float4 v = __ldcg(src + q * split4 + i4);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            out[i4] = acc;
            if (a.zexp) {
                const int q = (int)((beg + (size_t)i4 * 4) / r), kk = (int)((beg + (size_t)i4 * 4) % r);
                const int c = q - sh.q0c;
                int l = -1;
                for (int u = g0; u < g1; u++)
                    if (c >= s_cb[u] && c < s_ce[u]) l = s_sl[u];
                if (l >= 0) {
                    uint2 pk;
                    pk.x = (uint32_t)f32_to_bf16_rne(acc.x) | ((uint32_t)f32_to_bf16_rne(acc.y) << 16);
                    pk.y = (uint32_t)f32_to_bf16_rne(acc.z) | ((uint32_t)f32_to_bf16_rne(acc.w) << 16);
                    *reinterpret_cast<uint2*>(a.zexp + ((size_t)l * a.P + q) * rp + kk) = pk;
                }
            }
        }
        __threadfence();
        if (!rendezvous()) return false;
    }
    if (etid == 0) atomicAdd(a.zdone, 1);
    return true;
}

}  // namespace

}  // namespace moelora
