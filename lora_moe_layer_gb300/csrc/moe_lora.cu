// moe_lora.cu -- host side of the C ABI declared in include/moe_lora.h:
// argument validation, workspace layout, per-device kernel set-up and the
// launch sequence of one forward.
//
// One forward is five kernels on the caller's stream, chained with
// programmatic dependent launch so each can be resident before its
// predecessor drains (the blog's PDL step, "Efficiently serve dozens of
// fine-tuned models with vLLM ...", section "Execution optimizations"):
//   align -> gather x into bucket order
//         -> gate_up tcgen05 kernel (LoRA shrink items, then W1 tiles + expand, SiLU*up)
//         -> down tcgen05 kernel (LoRA shrink items, then W2 tiles + expand, x weight)
//         -> top-k reduce.
// A layer without adapters, or a batch without adapter tokens, has no shrink
// items (the blog's early exit, same section).
// Nothing here allocates device memory or synchronises the host.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.cuh"
#include "moe_lora.h"
#include "tma.cuh"

namespace moelora {
namespace {

constexpr int kDefaultBlockM = 16;
constexpr long kMaxZexpElems = 1L << 23;  // bf16 elements per zexp buffer (16 MiB)

// The expand's per-adapter width: r rounded up to 16, 32 or 64 (TMA reads zeros
// beyond r), with the swizzle whose span is one such row.
int expand_rpad_host(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : 64; }
CUtensorMapSwizzle expand_swizzle(int rp) {
    return rp == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : rp == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
}
// zexp columns: one r_pad-wide slot per adapter
long zexp_cols(int L, int r) { return (long)L * expand_rpad_host(r); }
constexpr int kMaxChunkMasks = 2048;  // 16 KiB of shared memory for the expand's chunk masks

struct Layout {
    int bm;
    int sms;  // SMs the split choices are planned for
    long P, NB, cap, tiles;
    // LoRA shrink plan: K-splits of the two shrinks, adapter buckets per task,
    // pairs per task, and the task-list bound
    int s1, s2, st_G, st_bn;
    long st_tasks_max;
    size_t hdr, sorted_ids, tile_expert, tile_lora, bucket_count, bucket_offset, compact_offset,
        compact_ids, active_experts, lora_buckets, hist, keys, align_sync, st_tasks, counters, z1, z1f, xc, act,
        z2, z2f, zexp1, zexp2, pair_out, tc_part, tc_counters, total;
    // LoRA expand on the tensor cores (zexp buffers bounded), else on CUDA cores
    bool tc_expand;
    // tensor-core GEMM plan (shared by the launch code and the workspace size):
    // chunk widths, K-splits, and whether wide chunks run on CTA pairs
    int bn_gu, bn_dn, ks_gu, ks_dn;
    bool pair_cta;   // the GEMMs run as CTA pairs (moe_gemm_2sm.cu)
    int ranks;       // CTAs per GEMM task: 2 with pair_cta, else 1
    int nu_gu, nu_dn;  // CTA pairs: weight rows per MMA chain of the two GEMMs
    int nt_gu, nt_dn;  // CTA pairs: the same for experts in chunks of 256 + 128 pairs
    bool w8;           // FP8 (E4M3) base weights: always the CTA-pair kernels
    long tiles_gu, tiles_dn;
    long nbl;  // upper bound of (expert, adapter >= 0) buckets with pairs
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

constexpr int kMaxDevices = 64;
constexpr int kFallbackSms = 152;  // GB300, when no device is visible (planning on a host without GPU)

// Multiprocessor count of the current device, looked up once per device (an
// attribute query: no context work, no allocation); kFallbackSms without one.
int current_device_sms() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return kFallbackSms;
    }
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return kFallbackSms;
    }
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// host-checkable validation; returns a status
int check_dims(const moe_lora_dims* d) {
    if (!d) return MOELORA_EINVAL;
    if (d->T < 0 || d->H <= 0 || d->I <= 0 || d->E <= 0 || d->k <= 0 || d->L < 0) return MOELORA_EINVAL;
    if (d->block_m != 0 && (!is_pow2(d->block_m) || d->block_m > 256)) return MOELORA_EINVAL;
    if (d->options & ~MOELORA_OPT_SINGLE_CTA) return MOELORA_EINVAL;
    if (d->sm_count < 0 || d->sm_count > 4096) return MOELORA_EINVAL;
    if (d->L > 0) {
        if (d->r <= 0) return MOELORA_EINVAL;
        if (d->r % 8 != 0 || d->r > 64) return MOELORA_EUNSUPPORTED;
    }
    if (d->H % 8 != 0 || d->I % 8 != 0) return MOELORA_EUNSUPPORTED;
    // index arithmetic of the kernels stays in int for these
    const long long P = (long long)d->T * d->k;
    const long long NB = (long long)d->E * (d->L + 1);
    if (P > (1LL << 28) || NB > (1LL << 22)) return MOELORA_EUNSUPPORTED;
    if ((long long)d->L * d->E * 64 > (1LL << 30)) return MOELORA_EUNSUPPORTED;
    const int bm = d->block_m ? d->block_m : kDefaultBlockM;
    const long long nonempty = std::min(NB, P);
    if (P + nonempty * (bm - 1) > (1LL << 30)) return MOELORA_EUNSUPPORTED;
    return MOELORA_OK;
}

// K-splits for a GEMM whose weight tiles alone would leave SMs idle: the
// smallest split count whose task count fills the kSms SMs' waves to >= 90%,
// keeping >= 512 K-elements per split.  The count only changes the balance,
// not the result.
int pick_ksplit(long tiles, int K, long kSms) {
    if (tiles >= 2 * kSms) return 1;
    int best = 1;
    double best_eff = 0.0;
    for (int ks = 1; ks <= 8 && K / ks >= 512; ks++) {
        const long tasks = tiles * ks;
        const long waves = (tasks + kSms - 1) / kSms;
        const double eff = (double)tasks / (double)(waves * kSms);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = ks;
        }
        if (eff >= 0.9) return ks;
    }
    return best;
}

// K-splits of a shrink.  Shrink items are taken ahead of the GEMM tasks, so
// when there are many shrink tasks (a quarter of the SMs or more),
// unsplit items about the size of a GEMM task keep the SMs balanced and skip
// the partial sums; with few (decode), the items are split so every SM takes a
// small share instead of a few SMs taking whole items.  At least two 64-wide K
// steps per split.
int pick_shrink_split(long est_tasks, int K, long kSms) {
    const int nkb = (K + 63) / 64;
    if (est_tasks * 4 >= kSms) return 1;
    const long want = (kSms + std::max<long>(est_tasks, 1) - 1) / std::max<long>(est_tasks, 1);
    return (int)std::max<long>(1, std::min<long>({want, (long)std::max(1, nkb / 2), 32L}));
}

// Shrink plan from the expected number of touched (expert, adapter) buckets
// when the pairs spread uniformly over the E*L of them.
void plan_shrinks(const moe_lora_dims* d, Layout* L) {
    if (d->L <= 0) {
        L->s1 = L->s2 = 0;
        L->st_G = L->st_bn = 0;
        L->st_tasks_max = 0;
        return;
    }
    // a shrink item stacks 128 / r buckets per CTA of its task
    L->st_G = L->ranks * (128 / d->r);
    // an item's pairs: one TMEM accumulator buffer of both one-CTA GEMM
    // kernels, or the 256 pair rows of a CTA pair
    const double nbl = (double)d->E * d->L;
    const double est_buckets = std::max(1.0, nbl * (1.0 - std::exp(-(double)L->P / nbl)));
    const long est_groups = std::max<long>(1, (long)std::ceil(est_buckets / L->st_G));
    const long rows_per_group = (L->P + est_groups - 1) / est_groups;
    L->st_bn = L->pair_cta ? 256 : std::min(2 * L->bn_gu, L->bn_dn);
    const long est_tasks = est_groups * ((rows_per_group + L->st_bn - 1) / L->st_bn);
    const long slots = std::max(1, L->sms / L->ranks);
    L->s1 = pick_shrink_split(est_tasks, d->H, slots);
    L->s2 = pick_shrink_split(est_tasks, d->I, slots);
    L->st_tasks_max = (L->nbl + L->st_G - 1) / L->st_G + (L->P + L->st_bn - 1) / L->st_bn;
}

// Expected distinct adapters among one expert's pairs (capped at a 256-pair
// chunk), with pairs spread evenly over experts and adapters drawn uniformly.
double expected_adapters_per_chunk(const moe_lora_dims* d, long P) {
    if (d->L <= 0 || P <= 0) return 0.0;
    const double experts = (double)std::max<long>(1, std::min<long>(d->E, P));
    const double pairs = std::min(256.0, (double)P / experts);
    return d->L * (1.0 - std::pow(1.0 - 1.0 / d->L, pairs));
}

// `rows` split into the fewest chains of at most `cap` rows, each a multiple of `mult`
int chain_rows_cap(long rows, long cap, long mult) {
    const long n = (rows + cap - 1) / cap;
    return (int)(((rows + n - 1) / n + mult - 1) / mult * mult);
}

// Weight rows per MMA chain of the CTA-pair kernel: the fewest chains of at
// most 256, each a multiple of 16 (2880 -> 12 x 240).
int chain_rows(long rows) { return chain_rows_cap(rows, 256, 16); }

// The same when the tasks are few (at most three rounds over the CTA pairs,
// e.g. one dense expert): the chain count whose rounds x rows copied per
// stage (128 pair rows + the chain rows) is smallest, since a last round
// that only some pairs run costs as much as a full one.  28672 rows on 76
// pairs: 150 chains of 192 (2 rounds) instead of 112 of 256 (2 rounds of
// larger stages).
int chain_rows_balanced(long rows, long chunks, long pairs) {
    const long n0 = (rows + 255) / 256;
    int best = chain_rows(rows);
    if (n0 * chunks > 3 * pairs) return best;
    long best_cost = (n0 * chunks + pairs - 1) / pairs * (128 + best);
    for (long n = n0 + 1; n <= (rows + 127) / 128; n++) {
        const int nu = (int)(((rows + n - 1) / n + 15) / 16 * 16);
        const long cost = (n * chunks + pairs - 1) / pairs * (128 + nu);
        if (cost < best_cost) {
            best_cost = cost;
            best = nu;
        }
    }
    return best;
}

// Weight rows per MMA chain for experts in chunks of 256 + 128 pairs, whose
// last 128 pairs have accumulators of 64 lanes x rows/2 columns per chain
// beside the main ones: the fewest chains of at most 160 rows (3 x 160 <= 512
// TMEM columns), each a multiple of 32 (2880 -> 18 x 160).
int chain_rows_tail(long rows) { return chain_rows_cap(rows, 160, 32); }

// Wide chunks (more than 48 pairs per expert on average) run on CTA pairs:
// chunks of 256 pairs, gate_up tasks of nu units (chains: their gate and
// their up rows), down tasks of 2 nu W2 rows, or, for experts the kernel
// finds cheaper that way, chunks of 256 + 128 pairs with chains of nu_t rows;
// as long as the pair kernel covers the layer (at most 64 adapters with the
// tensor-core expand, its chunk masks and zexp buffers within bounds, a ring
// that fits).
bool plan_pair_gemms(const moe_lora_dims* d, Layout* L, long experts_max, long avg_pairs) {
    if (d->L > 0 && (d->L > 64 || L->P * zexp_cols(d->L, d->r) > kMaxZexpElems)) return false;
    const long chunks = experts_max + (L->P + 255) / 256;
    if (d->L > 0 && chunks > kMaxChunkMasks) return false;
    if (tc2_plan_stages(d->E, d->L > 0 ? (int)chunks : 0) < 3) return false;
    L->pair_cta = true;
    L->ranks = 2;
    L->tc_expand = d->L > 0;
    L->bn_gu = L->bn_dn = 256;
    // gate_up takes no K split on CTA pairs, so its chain width balances the
    // rounds when the tasks are few; down balances them by its K split
    const long pairs = std::max(1, L->sms / 2), est_chunks = experts_max * ((avg_pairs + 255) / 256);
    L->nu_gu = chain_rows_balanced(d->I, est_chunks, pairs);
    L->nu_dn = chain_rows((d->H + 1) / 2);
    L->nt_gu = chain_rows_tail(d->I);
    L->nt_dn = chain_rows_tail((d->H + 1) / 2);
    // weight tiles per chunk in the two modes: the larger count bounds the
    // tasks; the split choice expects mode 0 (chunks of up to 256 pairs)
    const long nt_gu = (d->I + L->nu_gu - 1) / L->nu_gu, nt_dn = (d->H + 2 * L->nu_dn - 1) / (2 * L->nu_dn);
    const long ntt_gu = L->nt_gu ? (d->I + L->nt_gu - 1) / L->nt_gu : 0;
    const long ntt_dn = L->nt_dn ? (d->H + 2 * L->nt_dn - 1) / (2 * L->nt_dn) : 0;
    L->tiles_gu = std::max(nt_gu, ntt_gu) * chunks;
    L->tiles_dn = std::max(nt_dn, ntt_dn) * chunks;
    L->ks_gu = 1;
    L->ks_dn = pick_ksplit(nt_dn * est_chunks, d->I, pairs);
    return true;
}

// false: FP8 weights asked for a layer the CTA-pair kernels do not cover
bool plan_gemms(const moe_lora_dims* d, Layout* L) {
    const long experts_max = std::max<long>(1, std::min<long>(d->E, L->P));
    const long avg_pairs = L->P > 0 ? (L->P + experts_max - 1) / experts_max : 0;
    const bool narrow = avg_pairs <= 48;
    L->pair_cta = false;
    L->ranks = 1;
    L->nu_gu = L->nu_dn = 0;
    L->nt_gu = L->nt_dn = 0;
    // FP8 weights are dequantised in the CTA-pair kernels only, whatever the batch
    if (L->w8) return plan_pair_gemms(d, L, experts_max, std::max<long>(avg_pairs, 1));
    if (!narrow && !(d->options & MOELORA_OPT_SINGLE_CTA) && plan_pair_gemms(d, L, experts_max, avg_pairs)) return true;
    L->bn_gu = narrow ? 64 : 128;
    L->bn_dn = narrow ? 64 : 256;
    const long nt_gu = (d->I + 127) / 128, nt_dn = (d->H + 127) / 128;
    // upper bounds on the (expert, tile, chunk) count, for workspace sizing
    L->tiles_gu = nt_gu * (experts_max + (L->P + L->bn_gu - 1) / L->bn_gu);
    L->tiles_dn = nt_dn * (experts_max + (L->P + L->bn_dn - 1) / L->bn_dn);
    // expected counts with the pairs spread evenly, for the split choice
    const long est_gu = nt_gu * experts_max * ((avg_pairs + L->bn_gu - 1) / L->bn_gu);
    const long est_dn = nt_dn * experts_max * ((avg_pairs + L->bn_dn - 1) / L->bn_dn);
    L->ks_gu = pick_ksplit(est_gu, d->H, L->sms);
    L->ks_dn = pick_ksplit(est_dn, d->I, L->sms);
    return true;
}

int make_layout(const moe_lora_dims* d, Layout* L, bool w8 = false) {
    const int st = check_dims(d);
    if (st != MOELORA_OK) return st;
    // FP8 codes are TMA-copied with byte strides: rows of H and I codes must be
    // multiples of 16 bytes
    if (w8 && (d->H % 16 != 0 || d->I % 16 != 0)) return MOELORA_EUNSUPPORTED;
    L->w8 = w8;
    L->bm = d->block_m ? d->block_m : kDefaultBlockM;
    L->sms = d->sm_count > 0 ? d->sm_count : current_device_sms();
    L->P = (long)d->T * d->k;
    L->NB = (long)d->E * (d->L + 1);
    L->cap = L->P + std::min(L->NB, L->P) * (L->bm - 1);
    L->tiles = L->cap / L->bm;
    const int r = d->L > 0 ? d->r : 0;
    L->nbl = std::max<long>(std::min<long>((long)d->E * d->L, L->P), 1);
    // zexp: per pair, one r_pad-wide slot per adapter.  The tensor-core expand
    // pays one K block per group of a chunk's adapters; it is used when chunks
    // are expected to mix several adapters (the CUDA-core expand then reloads
    // B rows per adapter run) and while zexp stays small (it is rewritten
    // every forward).
    L->tc_expand = d->L > 0 && L->P * zexp_cols(d->L, d->r) <= kMaxZexpElems &&
                   expected_adapters_per_chunk(d, L->P) >= 4.0;
    if (!plan_gemms(d, L)) return MOELORA_EUNSUPPORTED;
    plan_shrinks(d, L);
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = up256(o + bytes); return at; };
    L->hdr = take(sizeof(WsHeader));
    L->sorted_ids = take(sizeof(int32_t) * std::max<long>(L->cap, 1));
    L->tile_expert = take(sizeof(int32_t) * std::max<long>(L->tiles, 1));
    L->tile_lora = take(sizeof(int32_t) * std::max<long>(L->tiles, 1));
    L->bucket_count = take(sizeof(int32_t) * L->NB);
    L->bucket_offset = take(sizeof(int32_t) * (L->NB + 1));
    L->compact_offset = take(sizeof(int32_t) * (L->NB + 1));
    L->compact_ids = take(sizeof(int32_t) * std::max<long>(L->P, 1));
    L->active_experts = take(sizeof(int32_t) * d->E);
    L->lora_buckets = take(sizeof(int32_t) * std::max<long>(std::min(L->NB, L->P), 1));
    L->hist = take(sizeof(int32_t) * align_hist_global_ints(d->E, d->L));
    L->keys = take(sizeof(int32_t) *
                   (align_keys_smem_bytes(d->E, d->L, L->P, kAlignRowsStable) ? 0 : std::max<long>(L->P, 1)));
    // the multi-CTA align's sync words and per-bucket counts
    L->align_sync = take(sizeof(int32_t) * (4 + L->NB));
    L->st_tasks = take(sizeof(int4) * std::max<long>(L->st_tasks_max, 1));
    // the two GEMMs' task counters, the split arrivals of the two shrinks'
    // tasks (per CTA of a task), then the two finished-task counts
    L->counters = take(sizeof(int32_t) * (2 + 2 * L->ranks * std::max<long>(L->st_tasks_max, 1) + 2));
    L->z1 = take(sizeof(float) * (size_t)(L->s1 > 1 ? L->s1 : 0) * L->P * r);
    L->z1f = take(sizeof(float) * (size_t)L->P * r);
    L->xc = take(sizeof(uint16_t) * (size_t)L->P * d->H);
    L->act = take(sizeof(uint16_t) * (size_t)L->P * d->I);
    L->z2 = take(sizeof(float) * (size_t)(L->s2 > 1 ? L->s2 : 0) * L->P * r);
    L->z2f = take(sizeof(float) * (size_t)L->P * r);
    const size_t zx = L->tc_expand ? sizeof(uint16_t) * (size_t)L->P * zexp_cols(d->L, d->r) : 0;
    L->zexp1 = take(zx);
    L->zexp2 = take(zx);
    // w * d per pair: bf16 [P][H] when the down GEMM does not split K (the
    // activation type, like the per-pair outputs the reduce sums), else one
    // fp32 [P][H] slab per K-split (partial sums stay exact until the reduce)
    L->pair_out = take(L->ks_dn > 1 ? sizeof(float) * (size_t)L->ks_dn * L->P * d->H
                                    : sizeof(uint16_t) * (size_t)L->P * d->H);
    const size_t part_gu = L->ks_gu > 1 ? (size_t)L->tiles_gu * L->ks_gu * 2 * L->bn_gu * 128 : 0;
    L->tc_part = take(sizeof(float) * part_gu);
    L->tc_counters = take(sizeof(int32_t) * (L->tiles_gu + L->tiles_dn));
    L->total = o;
    return MOELORA_OK;
}

struct DeviceInfo {
    int sms = 0;
    int pairs_gu = 0, pairs_dn = 0;  // co-resident CTA pairs of the two pair-GEMM kernels
    cudaError_t init_err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_once[kMaxDevices];

int device_setup(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOELORA_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MOELORA_EUNSUPPORTED;
    DeviceInfo* info = &g_dev[dev];
    std::call_once(g_once[dev], [info, dev]() {
        cudaError_t e = cudaDeviceGetAttribute(&info->sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = init_align_attributes();
        if (e == cudaSuccess) e = init_tc_attributes();
        if (e == cudaSuccess) e = init_tc2_attributes();
        if (e == cudaSuccess) {
            info->pairs_gu = tc2_max_pairs(true);
            info->pairs_dn = tc2_max_pairs(false);
        }
        info->init_err = e;
    });
    if (info->init_err != cudaSuccess) return MOELORA_ECUDA;
    *out = info;
    return MOELORA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// bf16 tiled tensor map (128-byte swizzle unless given), OOB elements read as zero
bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides_bytes, const cuuint32_t* box,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
                           strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// FP8 codes (one byte each), no swizzle (the converters read plain rows)
bool encode_u8_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), dims,
                           strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
// E4M3 codes of W1 [E][2I][H] as {H, I, 2, E} / W2 [E][H][I] as {I, H, E}:
// boxes of 64 codes (one K step) x rows
bool encode_w1q_map(CUtensorMap* map, const void* W1q, int E, int I, int H, int rows) {
    const cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
    const cuuint64_t strides[3] = {(cuuint64_t)H, (cuuint64_t)I * H, (cuuint64_t)2 * I * H};
    const cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, 1};
    return encode_u8_map(map, W1q, 4, dims, strides, box);
}
bool encode_w2q_map(CUtensorMap* map, const void* W2q, int E, int I, int H, int rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)E};
    const cuuint64_t strides[2] = {(cuuint64_t)I, (cuuint64_t)H * I};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    return encode_u8_map(map, W2q, 3, dims, strides, box);
}

// W1 [E][2I][H] viewed as [E][2][I][H]: boxes of 64 (K) x 128 units of one half
bool encode_w1_map(CUtensorMap* map, const void* W1, int E, int I, int H, int box_rows = 128) {
    const cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
    const cuuint64_t strides[3] = {(cuuint64_t)H * 2, (cuuint64_t)I * H * 2, (cuuint64_t)2 * I * H * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
    return encode_bf16_map(map, W1, 4, dims, strides, box);
}

// W2 [E][H][I]: boxes of 64 (K) x 128 rows (CTA pairs: half a chain)
bool encode_w2_map(CUtensorMap* map, const void* W2, int E, int I, int H, int box_rows = 128) {
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)E};
    const cuuint64_t strides[2] = {(cuuint64_t)I * 2, (cuuint64_t)H * I * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    return encode_bf16_map(map, W2, 3, dims, strides, box);
}

// adapter matrices A [L][E][r][K] as [L*E*r][K]: boxes of 64 (K) x r rows
bool encode_adapter_map(CUtensorMap* map, const void* A, int L, int E, int r, int K) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)L * E * r};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)r};
    return encode_bf16_map(map, A, 2, dims, strides, box);
}

// pair rows [P][K] (x in bucket order, or act): boxes of 64 (K) x box_rows
// rows (16 for decode-sized chunks, 64 for wide ones)
bool encode_rows_map(CUtensorMap* map, const void* rows, long P, int K, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)P};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    return encode_bf16_map(map, rows, 2, dims, strides, box);
}

// zexp [L][P][r_pad]: boxes of r_pad x rows pair rows x 64 / r_pad adapters
// (one ring stage's sub-tiles, adapter outermost)
bool encode_zexp_map(CUtensorMap* map, const void* zexp, long P, int L, int r, int rows, bool one_adapter = false) {
    const int rp = expand_rpad_host(r);
    const cuuint64_t dims[3] = {(cuuint64_t)rp, (cuuint64_t)P, (cuuint64_t)L};
    const cuuint64_t strides[2] = {(cuuint64_t)rp * 2, (cuuint64_t)P * rp * 2};
    const cuuint32_t box[3] = {(cuuint32_t)rp, (cuuint32_t)rows, one_adapter ? 1u : (cuuint32_t)(64 / rp)};
    return encode_bf16_map(map, zexp, 3, dims, strides, box, expand_swizzle(rp));
}
int pair_box_rows(int bn) { return bn >= 256 ? 256 : bn >= 128 ? 64 : 16; }  // matches the kernels' kRowsFor<BN>

// B1 [L][E][2I][r] as {r, I, 2, E, L}: boxes of r_pad (zeros beyond r) x 128
// units of one half x 64 / r_pad adapters (zeros beyond L); strides increase
// with the dimension, the swizzle span is one r_pad-wide row, and each
// adapter's 128 x r_pad tile lands after the previous one
bool encode_b1_map(CUtensorMap* map, const void* B1, int L, int E, int I, int r, bool one_adapter = false,
                   int box_rows = 128) {
    const int rp = expand_rpad_host(r);
    const cuuint64_t dims[5] = {(cuuint64_t)r, (cuuint64_t)I, 2, (cuuint64_t)E, (cuuint64_t)L};
    const cuuint64_t strides[4] = {(cuuint64_t)r * 2, (cuuint64_t)I * r * 2, (cuuint64_t)2 * I * r * 2,
                                   (cuuint64_t)E * 2 * I * r * 2};
    const cuuint32_t box[5] = {(cuuint32_t)rp, (cuuint32_t)box_rows, 1, 1, one_adapter ? 1u : (cuuint32_t)(64 / rp)};
    return encode_bf16_map(map, B1, 5, dims, strides, box, expand_swizzle(rp));
}

// B2 [L][E][H][r] as {r, H, E, L}: boxes of r_pad x 128 rows (CTA pairs: half a
// chain) x 64 / r_pad adapters
bool encode_b2_map(CUtensorMap* map, const void* B2, int L, int E, int H, int r, bool one_adapter = false,
                   int box_rows = 128) {
    const int rp = expand_rpad_host(r);
    const cuuint64_t dims[4] = {(cuuint64_t)r, (cuuint64_t)H, (cuuint64_t)E, (cuuint64_t)L};
    const cuuint64_t strides[3] = {(cuuint64_t)r * 2, (cuuint64_t)H * r * 2, (cuuint64_t)E * H * r * 2};
    const cuuint32_t box[4] = {(cuuint32_t)rp, (cuuint32_t)box_rows, 1, one_adapter ? 1u : (cuuint32_t)(64 / rp)};
    return encode_bf16_map(map, B2, 4, dims, strides, box, expand_swizzle(rp));
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// Workspace bytes that serve both forwards of these dims: the bf16 plan and,
// where the layer supports it, the FP8-weight plan (0 if the dims are invalid).
size_t workspace_need(const moe_lora_dims* d) {
    Layout L;
    if (make_layout(d, &L) != MOELORA_OK) return 0;
    size_t n = L.total;
    Layout L8;
    if (make_layout(d, &L8, true) == MOELORA_OK) n = std::max(n, L8.total);
    return n;
}

AlignArgs make_align_args(const moe_lora_dims* d, const Layout& L, const int32_t* topk_ids,
                          const int32_t* lora_ids, void* ws, int rows = kAlignRowsForward) {
    AlignArgs a = {};
    a.hist_rows = rows;
    a.T = d->T; a.k = d->k; a.E = d->E; a.L = d->L; a.bm = L.bm;
    a.topk_ids = topk_ids;
    a.lora_ids = lora_ids;
    a.sorted_ids = at<int32_t>(ws, L.sorted_ids);
    a.tile_expert = at<int32_t>(ws, L.tile_expert);
    a.tile_lora = at<int32_t>(ws, L.tile_lora);
    a.num_post_padded = nullptr;
    a.bucket_count = at<int32_t>(ws, L.bucket_count);
    a.bucket_offset = at<int32_t>(ws, L.bucket_offset);
    a.compact_offset = at<int32_t>(ws, L.compact_offset);
    a.compact_ids = at<int32_t>(ws, L.compact_ids);
    a.active_experts = at<int32_t>(ws, L.active_experts);
    a.lora_buckets = at<int32_t>(ws, L.lora_buckets);
    a.hist_global = align_hist_smem_bytes(d->E, d->L, rows) ? nullptr : at<int>(ws, L.hist);
    a.keys_in_smem = align_keys_smem_bytes(d->E, d->L, L.P, rows) ? 1 : 0;
    a.tabs_in_smem = align_tabs_smem_bytes(d->E, d->L, rows) ? 1 : 0;
    a.keys_global = a.keys_in_smem ? nullptr : at<int>(ws, L.keys);
    a.full_outputs = 0;
    a.zero_ints = at<int>(ws, L.counters);
    a.n_zero = 2 + (d->L > 0 ? (int)(2 * L.ranks * L.st_tasks_max + 2) : 0);
    a.st_tasks = d->L > 0 ? at<int4>(ws, L.st_tasks) : nullptr;
    a.st_G = L.st_G;
    a.st_BN = L.st_bn;
    a.zero_ints2 = at<int>(ws, L.tc_counters);
    a.n_zero2 = L.ks_gu > 1 ? (int)L.tiles_gu : 0;  // gate_up split arrivals (down splits write slabs)
    a.hdr = at<WsHeader>(ws, L.hdr);
    return a;
}

}  // namespace
}  // namespace moelora

using namespace moelora;

extern "C" {

MOELORA_API const char* moe_lora_strerror(int code) {
    switch (code) {
        case MOELORA_OK: return "ok";
        case MOELORA_EINVAL: return "invalid argument (null pointer or impossible size)";
        case MOELORA_ENOSPC: return "workspace smaller than moe_lora_workspace_bytes()";
        case MOELORA_EUNSUPPORTED: return "unsupported size or alignment (H, I multiples of 8; r multiple of 8 <= 64; 16-byte aligned pointers)";
        case MOELORA_ECUDA: return "a CUDA runtime call failed";
        case MOELORA_EDEVICE_ID: return "the device met an expert or adapter id out of range; those pairs were left out";
        case MOELORA_ETIMEOUT: return "a kernel gave up a bounded wait on its data pipeline; the result is incomplete";
        default: return "unknown status";
    }
}

MOELORA_API int moe_lora_version(void) { return 100; }

MOELORA_API int64_t moe_lora_align_capacity(const moe_lora_dims* d) {
    Layout L;
    const int st = make_layout(d, &L);
    return st == MOELORA_OK ? (int64_t)L.cap : (int64_t)st;
}

MOELORA_API size_t moe_lora_workspace_bytes(const moe_lora_dims* d) { return workspace_need(d); }

MOELORA_API int moe_lora_workspace_layout(const moe_lora_dims* d, moe_lora_ws_layout* out) {
    if (!out) return MOELORA_EINVAL;
    Layout L;
    const int st = make_layout(d, &L);
    if (st != MOELORA_OK) return st;
    const bool lora = d->L > 0;
    out->compact_ids = L.compact_ids;
    out->compact_offset = L.compact_offset;
    out->z1 = lora ? L.z1f : 0;
    out->act = L.act;
    out->z2 = lora ? L.z2f : 0;
    out->pair_out = L.pair_out;
    out->s1 = L.s1;
    out->s2 = L.s2;
    out->down_splits = std::max(1, L.ks_dn);
    out->launches = 5;  // align, gather, gate_up, down, reduce
    out->gemm_ctas = L.ranks;
    out->tc_expand = L.tc_expand ? 1 : 0;
    out->pair_out_bf16 = L.ks_dn > 1 ? 0 : 1;
    out->total = workspace_need(d);
    return MOELORA_OK;
}

MOELORA_API int moe_lora_align(const moe_lora_dims* d, const int32_t* topk_ids,
                               const int32_t* token_lora_ids, int32_t* sorted_ids,
                               int32_t* tile_expert, int32_t* tile_lora, int32_t* num_post_padded,
                               int32_t* bucket_count, int32_t* bucket_offset, void* workspace,
                               size_t workspace_bytes, void* stream) {
    Layout L;
    int st = make_layout(d, &L);
    if (st != MOELORA_OK) return st;
    if (!sorted_ids || !tile_expert || !tile_lora || !num_post_padded || !bucket_count ||
        !bucket_offset || !workspace)
        return MOELORA_EINVAL;
    if (d->T > 0 && (!topk_ids || !token_lora_ids)) return MOELORA_EINVAL;
    if (workspace_bytes < L.total || workspace_bytes < workspace_need(d)) return MOELORA_ENOSPC;
    if (!aligned16(workspace)) return MOELORA_EUNSUPPORTED;
    DeviceInfo* dev = nullptr;
    if ((st = device_setup(&dev)) != MOELORA_OK) return st;
    AlignArgs a = make_align_args(d, L, topk_ids, token_lora_ids, workspace, kAlignRowsStable);
    a.sorted_ids = sorted_ids;
    a.tile_expert = tile_expert;
    a.tile_lora = tile_lora;
    a.num_post_padded = num_post_padded;
    a.bucket_count = bucket_count;
    a.bucket_offset = bucket_offset;
    a.active_experts = nullptr;  // the standalone entry point skips the forward's work lists
    a.full_outputs = 1;
    const cudaError_t e = launch_align(a, align_smem_bytes(d->E, d->L, L.P, kAlignRowsStable), (cudaStream_t)stream);
    return e == cudaSuccess ? MOELORA_OK : MOELORA_ECUDA;
}

}  // extern "C"

namespace {

// Records event i (if given) just before kernel slot i of the forward; slot
// 5 is after the last kernel.  Skipped kernels still get their event.
struct Tracer {
    void* const* ev;
    int n;
    cudaStream_t s;
    bool ok = true;
    void mark(int i) {
        if (ev && i < n && ev[i] && cudaEventRecord((cudaEvent_t)ev[i], s) != cudaSuccess) ok = false;
    }
};

// FP8 base weights of a forward: E4M3 codes and per-output-row fp32 scales
struct W8Ptrs {
    const void* W1q;
    const float* W1s;
    const void* W2q;
    const float* W2s;
};

int forward_impl(const moe_lora_dims* d, const void* x, const int32_t* topk_ids,
                 const float* topk_weights, const int32_t* token_lora_ids, const void* W1,
                 const void* W2, const void* A1, const void* B1, const void* A2, const void* B2,
                 void* out, void* workspace, size_t workspace_bytes, void* stream,
                 void* const* events, int n_events, const W8Ptrs* w8 = nullptr) {
    Layout L;
    int st = make_layout(d, &L, w8 != nullptr);
    if (st != MOELORA_OK) return st;
    if (!workspace) return MOELORA_EINVAL;
    if (w8 ? !(w8->W1q && w8->W1s && w8->W2q && w8->W2s) : !(W1 && W2)) return MOELORA_EINVAL;
    if (w8) {
        const void* p8[] = {w8->W1q, w8->W2q, w8->W1s, w8->W2s};
        for (const void* p : p8)
            if (!aligned16(p)) return MOELORA_EUNSUPPORTED;
    }
    if (d->T > 0 && (!x || !topk_ids || !topk_weights || !token_lora_ids || !out)) return MOELORA_EINVAL;
    const bool has_lora = d->L > 0;
    if (has_lora && (!A1 || !B1 || !A2 || !B2)) return MOELORA_EINVAL;
    if (workspace_bytes < L.total || workspace_bytes < workspace_need(d)) return MOELORA_ENOSPC;
    const void* ptrs[] = {x, W1, W2, A1, B1, A2, B2, out, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MOELORA_EUNSUPPORTED;
    DeviceInfo* dev = nullptr;
    if ((st = device_setup(&dev)) != MOELORA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    void* ws = workspace;
    // programmatic dependent launch between the chained kernels; the legacy
    // NULL stream gets plain stream order
    const bool pdl = s != nullptr && s != cudaStreamLegacy;

    Tracer tr{events, n_events, s};
    AlignArgs aa = make_align_args(d, L, topk_ids, token_lora_ids, ws);
    tr.mark(0);
    {
        // batches of more than one CTA's pairs, at least 8 per bucket: the
        // multi-CTA align, its counts and sync words cleared first (its last
        // CTA scans all buckets alone, so many buckets favour the single-CTA
        // kernel); else the single-CTA kernel
        const int actas = align_multi_ctas(L.P, dev->sms);
        const int msmem =
            actas > 1 && L.P >= 8 * L.NB ? align_multi_smem_bytes(d->E, d->L, L.P, actas) : 0;
        if (msmem > 0) {
            aa.sync = at<int>(ws, L.align_sync);
            aa.gcount = aa.sync + 4;
            if (cudaMemsetAsync(aa.sync, 0, sizeof(int) * (4 + L.NB), s) != cudaSuccess ||
                launch_align_multi(aa, actas, msmem, s) != cudaSuccess)
                return MOELORA_ECUDA;
        } else if (launch_align(aa, align_smem_bytes(d->E, d->L, L.P, kAlignRowsForward), s) != cudaSuccess) {
            return MOELORA_ECUDA;
        }
    }
    if (d->T == 0) {
        for (int i = 1; i < MOELORA_TRACE_EVENTS; i++) tr.mark(i);
        return tr.ok ? MOELORA_OK : MOELORA_ECUDA;
    }

    WsHeader* hdr = at<WsHeader>(ws, L.hdr);
    const int sms = dev->sms;

    // x rows in bucket order: the B operand of the gate_up shrink and GEMM
    GatherArgs ga = {};
    ga.k = d->k; ga.H = d->H;
    ga.x = static_cast<const uint16_t*>(x);
    ga.compact_ids = at<int32_t>(ws, L.compact_ids);
    ga.hdr = hdr;
    ga.out = at<uint16_t>(ws, L.xc);
    if (L.tc_expand) {
        ga.zexp1 = at<uint16_t>(ws, L.zexp1);
        ga.zexp2 = at<uint16_t>(ws, L.zexp2);
        ga.zx_elems = L.P * zexp_cols(d->L, d->r);
    }
    tr.mark(1);
    {
        // warps per row: enough warps for 64 per SM, at most 8 per row
        ga.wpr = (int)std::max<long>(1, std::min<long>(8, (long)sms * 64 / std::max<long>(L.P, 1)));
        const int grid = (int)std::max<long>(1, std::min<long>((L.P * ga.wpr + 7) / 8, (long)sms * 8));
        if (launch_gather_rows(ga, grid, s, pdl) != cudaSuccess) return MOELORA_ECUDA;
    }

    TcArgs tc;
    memset(&tc, 0, sizeof(tc));
    tc.E = d->E; tc.L = d->L; tc.k = d->k; tc.r = has_lora ? d->r : 0; tc.I = d->I; tc.H = d->H;
    tc.P = (int)L.P;
    tc.lora_ids = token_lora_ids;
    tc.topk_weights = topk_weights;
    tc.active_experts = at<int32_t>(ws, L.active_experts);
    tc.compact_offset = at<int32_t>(ws, L.compact_offset);
    tc.compact_ids = at<int32_t>(ws, L.compact_ids);
    tc.hdr = hdr;
    tc.act_out = at<uint16_t>(ws, L.act);
    tc.pair_out = L.ks_dn > 1 ? at<float>(ws, L.pair_out) : nullptr;
    tc.pair_out16 = L.ks_dn > 1 ? nullptr : at<uint16_t>(ws, L.pair_out);
    int* task_counters = at<int>(ws, L.counters);  // gate_up, down; then the shrink counters
    int* sh_counters = task_counters + 2;
    tc.tc_expand = L.tc_expand ? 1 : 0;
    const long experts_bound = std::max<long>(1, std::min<long>(d->E, L.P));
    if (has_lora) {
        tc.sh_tasks = at<int4>(ws, L.st_tasks);
        tc.sh_G = L.st_G;
        tc.lora_buckets = at<int32_t>(ws, L.lora_buckets);
    }

    // wide chunks: both GEMMs on CTA pairs (moe_gemm_2sm.cu)
    const bool pc = L.pair_cta;

    // gate_up on the tensor cores: W1 tiles x (x rows in bucket order)
    {
        const int bn = L.bn_gu;
        tc.ksplit = L.ks_gu;
        tc.task_counter = task_counters;
        tc.part = at<float>(ws, L.tc_part);
        tc.tile_counters = at<int>(ws, L.tc_counters);
        tc.B = has_lora ? static_cast<const uint16_t*>(B1) : nullptr;
        tc.z = has_lora ? at<float>(ws, L.z1f) : nullptr;
        tc.zpart = at<float>(ws, L.z1);
        tc.sh_ks = L.s1;
        tc.sh_counters = sh_counters;
        tc.zdone = sh_counters + 2 * L.ranks * L.st_tasks_max;
        tc.zexp = L.tc_expand ? at<uint16_t>(ws, L.zexp1) : nullptr;
        tc.max_chunks = (int)(experts_bound + (L.P + bn - 1) / bn);
        tc.chunk_masks = L.tc_expand && d->L <= 64 && tc.max_chunks <= kMaxChunkMasks;
        if (pc) {
            // CTA pairs: 128 pair rows per CTA, chains of nu units (each CTA half of them)
            if (!tc.chunk_masks) tc.max_chunks = 0;
            tc.nu = L.nu_gu;
            tc.nu_t = L.nt_gu;
            const int half = L.nu_gu / 2, half_t = L.nt_gu / 2;
            if (w8) {
                tc.w8 = 1;
                tc.wscale = w8->W1s;
                tc.nstages = tc2_plan_stages_w8(d->E, tc.max_chunks);
                if (tc.nstages < 2) return MOELORA_EUNSUPPORTED;
                if (!encode_w1q_map(&tc.w8map, w8->W1q, d->E, d->I, d->H, half) ||
                    (half_t && !encode_w1q_map(&tc.w8map_t, w8->W1q, d->E, d->I, d->H, half_t)))
                    return MOELORA_ECUDA;
            } else {
                tc.nstages = tc2_plan_stages(d->E, tc.max_chunks);
                if (tc.nstages < 3) return MOELORA_EUNSUPPORTED;
            }
            if ((!w8 && (!encode_w1_map(&tc.wmap, W1, d->E, d->I, d->H, half) ||
                         (half_t && !encode_w1_map(&tc.wmap_t, W1, d->E, d->I, d->H, half_t)))) ||
                !encode_rows_map(&tc.xmap, at<uint16_t>(ws, L.xc), L.P, d->H, 128) ||
                (half_t && !encode_rows_map(&tc.xmap_t, at<uint16_t>(ws, L.xc), L.P, d->H, 64)) ||
                (has_lora && !encode_adapter_map(&tc.amap, A1, d->L, d->E, d->r, d->H)) ||
                (L.tc_expand && (!encode_b1_map(&tc.bmap, B1, d->L, d->E, d->I, d->r, false, half) ||
                                 (half_t && !encode_b1_map(&tc.bmap_t, B1, d->L, d->E, d->I, d->r, false, half_t)) ||
                                 !encode_zexp_map(&tc.zxmap, tc.zexp, L.P, d->L, d->r, 128) ||
                                 (half_t && !encode_zexp_map(&tc.zxmap_t, tc.zexp, L.P, d->L, d->r, 64)))))
                return MOELORA_ECUDA;
        } else {
            tc.nstages = tc_plan_stages(true, bn, tc.r, d->E, L.tc_expand, tc.chunk_masks ? tc.max_chunks : 0);
            if (tc.nstages < 2) return MOELORA_EUNSUPPORTED;
            const int rows = pair_box_rows(bn);
            if (!encode_w1_map(&tc.wmap, W1, d->E, d->I, d->H) ||
                !encode_rows_map(&tc.xmap, at<uint16_t>(ws, L.xc), L.P, d->H, rows) ||
                (has_lora && !encode_adapter_map(&tc.amap, A1, d->L, d->E, d->r, d->H)) ||
                (L.tc_expand && (!encode_b1_map(&tc.bmap, B1, d->L, d->E, d->I, d->r) ||
                                 !encode_b1_map(&tc.bmap1, B1, d->L, d->E, d->I, d->r, true) ||
                                 !encode_zexp_map(&tc.zxmap, tc.zexp, L.P, d->L, d->r, bn) ||
                                 !encode_zexp_map(&tc.zxmap1, tc.zexp, L.P, d->L, d->r, bn, true))))
                return MOELORA_ECUDA;
        }
        const long tasks = L.tiles_gu * L.ks_gu + L.st_tasks_max * L.s1;
        tr.mark(2);
        if (pc) {
            if (dev->pairs_gu < 1) return MOELORA_EUNSUPPORTED;
            const int grid = 2 * (int)std::max<long>(1, std::min<long>(tasks, dev->pairs_gu));
            if (launch_moe_gemm_2sm(tc, true, grid, s, pdl) != cudaSuccess) return MOELORA_ECUDA;
        } else {
            const int grid = (int)std::max<long>(1, std::min<long>(tasks, sms));
            if (launch_moe_gemm_tc(tc, true, bn, grid, s, pdl) != cudaSuccess) return MOELORA_ECUDA;
        }
    }

    // down on the tensor cores: W2 tiles x act rows
    {
        const int bn = L.bn_dn;
        tc.ksplit = L.ks_dn;
        tc.task_counter = task_counters + 1;
        tc.tile_counters = at<int>(ws, L.tc_counters) + L.tiles_gu;
        tc.B = has_lora ? static_cast<const uint16_t*>(B2) : nullptr;
        tc.z = has_lora ? at<float>(ws, L.z2f) : nullptr;
        tc.zpart = at<float>(ws, L.z2);
        tc.sh_ks = L.s2;
        tc.sh_counters = sh_counters + L.ranks * L.st_tasks_max;
        tc.zdone = sh_counters + 2 * L.ranks * L.st_tasks_max + 1;
        tc.zexp = L.tc_expand ? at<uint16_t>(ws, L.zexp2) : nullptr;
        tc.pair_split = (size_t)L.P * d->H;
        tc.max_chunks = (int)(experts_bound + (L.P + bn - 1) / bn);
        tc.chunk_masks = L.tc_expand && d->L <= 64 && tc.max_chunks <= kMaxChunkMasks;
        if (pc) {
            // CTA pairs: 128 act rows per CTA, two chains of nu W2 rows (each CTA half of each)
            if (!tc.chunk_masks) tc.max_chunks = 0;
            tc.nu = L.nu_dn;
            tc.nu_t = L.nt_dn;
            const int half = L.nu_dn / 2, half_t = L.nt_dn / 2;
            if (w8) {
                tc.w8 = 1;
                tc.wscale = w8->W2s;
                tc.nstages = tc2_plan_stages_w8(d->E, tc.max_chunks);
                if (tc.nstages < 2) return MOELORA_EUNSUPPORTED;
                if (!encode_w2q_map(&tc.w8map, w8->W2q, d->E, d->I, d->H, half) ||
                    (half_t && !encode_w2q_map(&tc.w8map_t, w8->W2q, d->E, d->I, d->H, half_t)))
                    return MOELORA_ECUDA;
            } else {
                tc.nstages = tc2_plan_stages(d->E, tc.max_chunks);
                if (tc.nstages < 3) return MOELORA_EUNSUPPORTED;
            }
            if ((!w8 && (!encode_w2_map(&tc.wmap, W2, d->E, d->I, d->H, half) ||
                         (half_t && !encode_w2_map(&tc.wmap_t, W2, d->E, d->I, d->H, half_t)))) ||
                !encode_rows_map(&tc.xmap, at<uint16_t>(ws, L.act), L.P, d->I, 128) ||
                (half_t && !encode_rows_map(&tc.xmap_t, at<uint16_t>(ws, L.act), L.P, d->I, 64)) ||
                (has_lora && !encode_adapter_map(&tc.amap, A2, d->L, d->E, d->r, d->I)) ||
                (L.tc_expand && (!encode_b2_map(&tc.bmap, B2, d->L, d->E, d->H, d->r, false, half) ||
                                 (half_t && !encode_b2_map(&tc.bmap_t, B2, d->L, d->E, d->H, d->r, false, half_t)) ||
                                 !encode_zexp_map(&tc.zxmap, tc.zexp, L.P, d->L, d->r, 128) ||
                                 (half_t && !encode_zexp_map(&tc.zxmap_t, tc.zexp, L.P, d->L, d->r, 64)))))
                return MOELORA_ECUDA;
        } else {
            tc.nstages = tc_plan_stages(false, bn, tc.r, d->E, L.tc_expand, tc.chunk_masks ? tc.max_chunks : 0);
            if (tc.nstages < 2) return MOELORA_EUNSUPPORTED;
            const int rows = pair_box_rows(bn);
            if (!encode_w2_map(&tc.wmap, W2, d->E, d->I, d->H) ||
                !encode_rows_map(&tc.xmap, at<uint16_t>(ws, L.act), L.P, d->I, rows) ||
                (has_lora && !encode_adapter_map(&tc.amap, A2, d->L, d->E, d->r, d->I)) ||
                (L.tc_expand && (!encode_b2_map(&tc.bmap, B2, d->L, d->E, d->H, d->r) ||
                                 !encode_b2_map(&tc.bmap1, B2, d->L, d->E, d->H, d->r, true) ||
                                 !encode_zexp_map(&tc.zxmap, tc.zexp, L.P, d->L, d->r, bn) ||
                                 !encode_zexp_map(&tc.zxmap1, tc.zexp, L.P, d->L, d->r, bn, true))))
                return MOELORA_ECUDA;
        }
        const long tasks = L.tiles_dn * L.ks_dn + L.st_tasks_max * L.s2;
        tr.mark(3);
        if (pc) {
            if (dev->pairs_dn < 1) return MOELORA_EUNSUPPORTED;
            const int grid = 2 * (int)std::max<long>(1, std::min<long>(tasks, dev->pairs_dn));
            if (launch_moe_gemm_2sm(tc, false, grid, s, pdl) != cudaSuccess) return MOELORA_ECUDA;
        } else {
            const int grid = (int)std::max<long>(1, std::min<long>(tasks, sms));
            if (launch_moe_gemm_tc(tc, false, bn, grid, s, pdl) != cudaSuccess) return MOELORA_ECUDA;
        }
    }

    ReduceArgs ra = {};
    ra.T = d->T; ra.k = d->k; ra.H = d->H; ra.E = d->E; ra.L = d->L;
    ra.pair_out = L.ks_dn > 1 ? at<float>(ws, L.pair_out) : nullptr;
    ra.pair_out16 = L.ks_dn > 1 ? nullptr : at<uint16_t>(ws, L.pair_out);
    ra.nsplit = std::max(1, L.ks_dn);
    ra.split_stride = (size_t)L.P * d->H;
    ra.topk_ids = topk_ids;
    ra.lora_ids = token_lora_ids;
    ra.out = static_cast<uint16_t*>(out);
    tr.mark(4);
    {
        const long n = (long)d->T * (d->H / (ra.pair_out16 ? 8 : 4));  // hidden elements per thread
        const int grid = (int)std::max<long>(1, std::min<long>((n + 255) / 256, (long)sms * 8));
        if (launch_reduce(ra, grid, s, pdl) != cudaSuccess) return MOELORA_ECUDA;
    }
    tr.mark(5);
    return tr.ok ? MOELORA_OK : MOELORA_ECUDA;
}

}  // namespace

extern "C" {

MOELORA_API int moe_lora_forward(const moe_lora_dims* d, const void* x, const int32_t* topk_ids,
                                 const float* topk_weights, const int32_t* token_lora_ids,
                                 const void* W1, const void* W2, const void* A1, const void* B1,
                                 const void* A2, const void* B2, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    return forward_impl(d, x, topk_ids, topk_weights, token_lora_ids, W1, W2, A1, B1, A2, B2, out,
                        workspace, workspace_bytes, stream, nullptr, 0);
}

MOELORA_API int moe_lora_forward_w8(const moe_lora_dims* d, const void* x, const int32_t* topk_ids,
                                    const float* topk_weights, const int32_t* token_lora_ids,
                                    const void* W1q, const float* W1s, const void* W2q, const float* W2s,
                                    const void* A1, const void* B1, const void* A2, const void* B2, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    const W8Ptrs w8 = {W1q, W1s, W2q, W2s};
    return forward_impl(d, x, topk_ids, topk_weights, token_lora_ids, nullptr, nullptr, A1, B1, A2, B2, out,
                        workspace, workspace_bytes, stream, nullptr, 0, &w8);
}

MOELORA_API int moe_lora_forward_traced(const moe_lora_dims* d, const void* x,
                                        const int32_t* topk_ids, const float* topk_weights,
                                        const int32_t* token_lora_ids, const void* W1,
                                        const void* W2, const void* A1, const void* B1,
                                        const void* A2, const void* B2, void* out, void* workspace,
                                        size_t workspace_bytes, void* stream,
                                        void* const* kernel_events, int32_t n_events) {
    if (!kernel_events || n_events < MOELORA_TRACE_EVENTS) return MOELORA_EINVAL;
    return forward_impl(d, x, topk_ids, topk_weights, token_lora_ids, W1, W2, A1, B1, A2, B2, out,
                        workspace, workspace_bytes, stream, kernel_events, n_events);
}

MOELORA_API int moe_lora_forward_w8_traced(const moe_lora_dims* d, const void* x, const int32_t* topk_ids,
                                           const float* topk_weights, const int32_t* token_lora_ids,
                                           const void* W1q, const float* W1s, const void* W2q, const float* W2s,
                                           const void* A1, const void* B1, const void* A2, const void* B2,
                                           void* out, void* workspace, size_t workspace_bytes, void* stream,
                                           void* const* kernel_events, int32_t n_events) {
    if (!kernel_events || n_events < MOELORA_TRACE_EVENTS) return MOELORA_EINVAL;
    const W8Ptrs w8 = {W1q, W1s, W2q, W2s};
    return forward_impl(d, x, topk_ids, topk_weights, token_lora_ids, nullptr, nullptr, A1, B1, A2, B2, out,
                        workspace, workspace_bytes, stream, kernel_events, n_events, &w8);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward without any allocation.
//
// Some callers cannot obtain device memory for a workspace: code running where
// cudaMalloc is off limits (it can block until the device is idle, so
// latency-critical or real-time loops avoid it), plugins whose host framework
// owns all device memory and exposes no allocator to them, or a caller with no
// allocator of its own at all.  For them the forward can run on a scratch
// buffer that lives inside this library: a file-scope array in device memory
// of kNoAllocScratchBytes bytes, which every GPU that loads the library holds
// until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = MOELORA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device.  In host code the array's
// name is only a host-side stand-in, so the address must come from the
// runtime; it is looked up once per device, with that device current.
void* g_noalloc_ptr[kMaxDevices];
cudaError_t g_noalloc_err[kMaxDevices];
std::once_flag g_noalloc_once[kMaxDevices];

}  // namespace

extern "C" {

MOELORA_API int moe_lora_forward_noalloc(const moe_lora_dims* d, const void* x,
                                         const int32_t* topk_ids, const float* topk_weights,
                                         const int32_t* token_lora_ids, const void* W1,
                                         const void* W2, const void* A1, const void* B1,
                                         const void* A2, const void* B2, void* out,
                                         void* stream) {
    // host-side checks first, so a refused call touches no CUDA state
    Layout L;
    const int st = make_layout(d, &L);
    if (st != MOELORA_OK) return st;
    if (!W1 || !W2) return MOELORA_EINVAL;
    if (d->T > 0 && (!x || !topk_ids || !topk_weights || !token_lora_ids || !out)) return MOELORA_EINVAL;
    if (d->L > 0 && (!A1 || !B1 || !A2 || !B2)) return MOELORA_EINVAL;
    if (workspace_need(d) > kNoAllocScratchBytes) return MOELORA_ENOSPC;  // needs more than the built-in scratch

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOELORA_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MOELORA_EUNSUPPORTED;
    std::call_once(g_noalloc_once[dev], [dev]() {
        g_noalloc_err[dev] = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch);
    });
    if (g_noalloc_err[dev] != cudaSuccess || g_noalloc_ptr[dev] == nullptr) return MOELORA_ECUDA;
    // The forward overwrites every scratch byte it later reads (the status word
    // and histograms are reset by its first kernel), so the previous call's
    // leftovers need no clearing.
    return forward_impl(d, x, topk_ids, topk_weights, token_lora_ids, W1, W2, A1, B1, A2, B2, out,
                        g_noalloc_ptr[dev], kNoAllocScratchBytes, stream, nullptr, 0);
}

MOELORA_API int moe_lora_selftest_wait(int32_t kind, void* workspace, void* stream) {
    if ((kind != 0 && kind != 1) || !workspace) return MOELORA_EINVAL;
    if (!aligned16(workspace)) return MOELORA_EUNSUPPORTED;
    return launch_selftest_wait(kind, workspace, (cudaStream_t)stream) == cudaSuccess ? MOELORA_OK : MOELORA_ECUDA;
}

MOELORA_API int moe_lora_get_status(const void* workspace, void* stream) {
    if (!workspace) return MOELORA_EINVAL;
    int32_t status = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&status, workspace, sizeof(status), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return MOELORA_ECUDA;
    }
    if (status == 0) return MOELORA_OK;
    return (status & (kStatusBadExpert | kStatusBadLora)) ? MOELORA_EDEVICE_ID : MOELORA_ETIMEOUT;
}

}  // extern "C"
