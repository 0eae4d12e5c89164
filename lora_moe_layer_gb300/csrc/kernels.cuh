// kernels.cuh -- argument blocks and host launchers of the libmoelora kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moelora {

// ---------------------------------------------------------------- align ----
constexpr int kAlignMaxSmemHist = 160 * 1024;
constexpr int kAlignMaxSmem = 200 * 1024;  // histogram + pair keys

struct AlignArgs {
    int T, k, E, L, bm;
    const int32_t* topk_ids;   // [T*k]
    const int32_t* lora_ids;   // [T]
    // outputs
    int32_t* sorted_ids;       // [capacity]
    int32_t* tile_expert;      // [capacity / bm]
    int32_t* tile_lora;        // [capacity / bm]
    int32_t* num_post_padded;  // [1] or null
    int32_t* bucket_count;     // [NB]
    int32_t* bucket_offset;    // [NB + 1] padded starts
    int32_t* compact_offset;   // [NB + 1] unpadded starts
    int32_t* compact_ids;      // [P] pair of each compact row
    int32_t* active_experts;   // [E] or null (then the two lists below are skipped)
    int32_t* lora_buckets;     // [min(NB, P)]
    int* hist_global;          // [16 * NB] when the histogram does not fit in shared memory, else null
    int* zero_ints;            // [n_zero] cleared for the kernels that follow (shrink counters), or null
    int n_zero;
    int* zero_ints2;           // [n_zero2] second region (GEMM split-K counters), or null
    int n_zero2;
    // LoRA shrink task list (null: none): buckets of lora_buckets in groups of
    // st_G, each group's rows in chunks of at most st_BN, as (group, first row, rows, 0)
    int4* st_tasks;
    int st_G, st_BN;
    int* keys_global;          // [P] pair keys when they do not fit in shared memory
    int keys_in_smem;          // 1: keys in shared memory
    int tabs_in_smem;          // 1: bucket sizes and offsets also in shared memory
    int full_outputs;          // 1: also sentinels and per-tile expert/adapter (standalone align)
    int hist_rows;             // rows of NB ints in the histogram (kAlignRowsStable / kAlignRowsForward)
    WsHeader* hdr;
    // multi-CTA forward align: per-bucket counts and three sync words
    // (arrivals, offsets ready, OR of the bad-id bits), zeroed before the launch
    int* gcount;               // [NB]
    int* sync;                 // [4]
};

// histogram rows of the single-CTA align: per-warp counts for the standalone
// entry point (kAlignWarps rows), counts + lists for the forward
constexpr int kAlignRowsStable = 16;
constexpr int kAlignRowsForward = 3;
int align_hist_smem_bytes(int E, int L, int rows);  // 0 if the histogram must live in global memory
int align_keys_smem_bytes(int E, int L, long P, int rows);  // 0 if the pair keys must live in global memory
int align_tabs_smem_bytes(int E, int L, int rows);  // 0 if the bucket tables stay in global memory only
int align_smem_bytes(int E, int L, long P, int rows);  // dynamic shared memory of the align launch
long align_hist_global_ints(int E, int L);          // global histogram ints (stable rows) when it does not fit
cudaError_t launch_align(const AlignArgs& args, int smem_bytes, cudaStream_t stream);
// The forward's align on several CTAs (pairs in any order inside a bucket):
// 0 bytes if the bucket tables do not fit its shared memory (then the
// single-CTA kernel runs), and the CTA count for P pairs on `sms` SMs.
int align_multi_smem_bytes(int E, int L, long P, int ctas);
int align_multi_ctas(long P, int sms);
cudaError_t launch_align_multi(const AlignArgs& args, int ctas, int smem_bytes, cudaStream_t stream);
cudaError_t init_align_attributes();

// ------------------------------------------------------------ tcgen05 GEMM ----
// Grouped expert GEMM on the tensor cores (moe_gemm_tc.cu), weight rows on M.
constexpr int kTcSmemLimit = 227 * 1024 - 1024;
struct TcArgs {
    CUtensorMap wmap;            // W1 as [E][2][I][H] (gate_up) or W2 [E][H][I]; box 64 (K) x 128 rows
    CUtensorMap xmap;            // pair rows: x in bucket order [P][H] or act [P][I]; box 64 x 16, 64 or 256 rows
    CUtensorMap amap;            // LoRA A (A1 / A2) as [L*E*r][K]; box 64 (K) x r rows
    CUtensorMap bmap;            // LoRA B: B1 as {r, I, 2, E, L} / B2 as {r, H, E, L}; box r_pad x 128 rows x 64/r_pad adapters
    CUtensorMap bmap1;           // the same LoRA B with a one-adapter box
    CUtensorMap zxmap;           // zexp [L][P][r_pad] bf16; box r_pad x BN rows x 64/r_pad adapters
    CUtensorMap zxmap1;          // the same zexp with a one-adapter box
    int E, L, k, r, I, H, P;
    const uint16_t* B;           // B1 / B2 (null: no LoRA)
    float* z;                    // shrink output [P][r], written by the shrink items (null: no LoRA)
    // LoRA shrink items, run first (the GEMM epilogues wait for all of them):
    // align's task list, G adapter buckets per task, K-split into sh_ks parts
    const int4* sh_tasks;
    int sh_G, sh_ks;
    const int32_t* lora_buckets;
    float* zpart;                // [sh_ks][P][r] split partials (sh_ks > 1)
    int* sh_counters;            // [tasks] split arrivals, zeroed by align
    int* zdone;                  // shrink tasks finished, zeroed by align
    int tc_expand;               // 1: LoRA expand as extra tensor-core K-blocks; 0: CUDA cores in the epilogue
    uint16_t* zexp;              // [L][P][r_pad] bf16: z of each pair under its own adapter, zeros elsewhere
    int chunk_masks;             // 1: per-(expert, pair chunk) adapter masks in shared memory (L <= 64)
    int max_chunks;              // bound on (expert, pair chunk) count, for the mask table
    const int32_t* lora_ids;
    const float* topk_weights;
    const int32_t* active_experts;
    const int32_t* compact_offset;
    const int32_t* compact_ids;
    WsHeader* hdr;
    uint16_t* act_out;           // gate_up: [P][I] bf16
    float* pair_out;             // down, split K: [ksplit][P][H] fp32 by pair id, one slab per K-split
    uint16_t* pair_out16;        // down, one split: [P][H] bf16 by pair id (then pair_out is unused)
    size_t pair_split;           // down: elements between two K-splits' slabs (P * H)
    int nstages;
    int ksplit;                  // K-splits per weight tile (1: none)
    float* part;                 // gate_up split-K partial tiles [tiles][ksplit][acc columns][128]
    int* tile_counters;          // [tiles] split arrivals, zeroed by align
    int* task_counter;           // next task to take (each CTA takes its next one when it is ready for
                                 // it), zeroed by align; null: tasks dealt round-robin over the CTAs
    int nu;                      // CTA-pair kernel: weight rows per MMA chain (multiple of 16, <= 256)
    // CTA-pair kernel, experts whose pairs run in chunks of 256 + 128 (the
    // last 128 on an M = 128 MMA sharing the weight stage): chains of nu_t
    // rows (multiple of 32, <= 160; 0: no such chunks), and the maps with the
    // boxes of those tasks (pair rows and zexp 64 rows, weight and B rows nu_t / 2)
    int nu_t;
    CUtensorMap xmap_t, wmap_t, bmap_t, zxmap_t, w8map_t;
    // CTA-pair kernel with FP8 base weights: E4M3 codes of W1 as {H, I, 2, E}
    // / W2 as {I, H, E}, box 64 codes x nu/2 rows; one fp32 scale per output
    // row (W1s [E][2I] / W2s [E][H])
    CUtensorMap w8map;
    const float* wscale;
    int w8;
};
int tc_smem_bytes(bool gate_up, int bn, int r, int E, int nstages, bool tc_expand, int mask_chunks);
int tc_plan_stages(bool gate_up, int bn, int r, int E, bool tc_expand, int mask_chunks);
cudaError_t init_tc_attributes();
cudaError_t launch_moe_gemm_tc(const TcArgs& args, bool gate_up, int bn, int grid, cudaStream_t stream, bool pdl);
// The same GEMMs for wide pair chunks on CTA pairs (moe_gemm_2sm.cu): M = 256
// pair rows over the pair (chunks of up to 256 pairs, or 256 + 128 with chains
// of nu_t rows), two chains of nu weight rows, tensor-core expand only, chunk
// masks required, gate_up without K split.
int tc2_smem_bytes(int E, int nstages, int max_chunks, bool w8 = false);
int tc2_plan_stages(int E, int max_chunks);
// FP8 base weights: ring stages (pair rows, and the chain rows the codes are
// expanded into), 0 if fewer than two fit
int tc2_plan_stages_w8(int E, int max_chunks);
cudaError_t init_tc2_attributes();
int tc2_max_pairs(bool gate_up);  // co-resident pairs (0: none or query failed)
cudaError_t launch_moe_gemm_2sm(const TcArgs& args, bool gate_up, int grid, cudaStream_t stream, bool pdl);

struct GatherArgs {
    int k, H;
    const uint16_t* x;           // [T][H]
    const int32_t* compact_ids;
    const WsHeader* hdr;
    uint16_t* out;               // [P][H] rows in bucket order
    int wpr;                     // warps per row (1 .. 8)
    uint16_t* zexp1;             // [zx_elems] zeroed here (null: none)
    uint16_t* zexp2;
    long zx_elems;
};
cudaError_t launch_gather_rows(const GatherArgs& args, int grid, cudaStream_t stream, bool pdl);

// --------------------------------------------------------------- reduce ----
constexpr int kMaxSplitSlabs = 8;  // the host plans at most 8 K-splits per GEMM
struct ReduceArgs {
    int T, k, H, E, L;
    const float* pair_out;       // [nsplit][P][H]: the down GEMM's K-split slabs (fp32)
    const uint16_t* pair_out16;  // or, when the down GEMM does not split K, its [P][H] bf16 output
    int nsplit;                  // 1 .. kMaxSplitSlabs
    size_t split_stride;         // elements between slabs
    const int32_t* topk_ids;
    const int32_t* lora_ids;
    uint16_t* out;               // [T][H]
};
cudaError_t launch_reduce(const ReduceArgs& args, int grid, cudaStream_t stream, bool pdl);

// ------------------------------------------------------------- self-test ----
// one kernel whose wait nothing satisfies (kind 0: mbarrier phase, 1: counter)
cudaError_t launch_selftest_wait(int kind, void* workspace, cudaStream_t stream);

// common launch helper: optional programmatic-dependent-launch attribute
template <typename Kern, typename Args>
cudaError_t launch_k(Kern kernel, dim3 grid, dim3 block, int smem, cudaStream_t stream, bool pdl,
                     const Args& args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace moelora
