// kernels.cuh -- argument blocks and host launchers of the libmoelora kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moelora {

// ---------------------------------------------------------------- align ----
constexpr int kAlignMaxSmemHist = 160 * 1024;

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
    int32_t* scan_tmp;         // [max(E, NB) + 1]
    int* hist_global;          // [16 * NB] when the histogram does not fit in shared memory, else null
    WsHeader* hdr;
};

int align_hist_smem_bytes(int E, int L);   // 0 if the histogram must live in global memory
long align_hist_global_ints(int E, int L);
cudaError_t launch_align(const AlignArgs& args, int smem_bytes, cudaStream_t stream);
cudaError_t init_align_attributes();

// --------------------------------------------------------------- shrink ----
// z[s][row][0:r] = sum over the s-th K-split of A[l][e][0:r][k] * in(row)[k]
// for every compact row of every (e, l >= 0) bucket.
struct ShrinkArgs {
    int E, L, k, r, K, P;
    int S;                      // K-splits
    int in_is_x;                // 1: in(row) = x[compact_ids[row] / k]; 0: in(row) = act[row]
    const uint16_t* in;         // x [T][K] or act [P][K]
    const uint16_t* A;          // [L][E][r][K]
    const int32_t* lora_buckets;
    const int32_t* compact_offset;
    const int32_t* compact_ids;
    const WsHeader* hdr;
    float* z;                   // [S][P][r]
    int max_items;              // upper bound of buckets * S (host-known)
};
constexpr int kShrinkKC = 512;  // K elements per split
cudaError_t launch_shrink(const ShrinkArgs& args, int grid, cudaStream_t stream, bool pdl);
cudaError_t init_shrink_attributes();
int shrink_blocks_per_sm();

// ----------------------------------------------------------------- gemv ----
// Grouped GEMV over the active experts.  gate_up: act[row][i] =
// SiLU(g_i) * g_{I+i} with g = W1[e] x + B1[l][e] z1.  down: pair_out[p][h]
// = w_p * (W2[e] act[row] + B2[l][e] z2).
struct GemvArgs {
    int E, L, k, r, I, H, P;
    int gate_up;                 // 1: gate_up (+ SiLU*mul), 0: down (+ weight)
    const uint16_t* in;          // gate_up: x [T][H]; down: act [P][I]
    const uint16_t* W;           // W1 [E][2I][H] or W2 [E][H][I]
    const uint16_t* B;           // B1 [L][E][2I][r] or B2 [L][E][H][r] (null: no LoRA)
    const float* zpart;          // [S][P][r] shrink partials (null: no LoRA)
    int S;
    const int32_t* lora_ids;     // [T]
    const float* topk_weights;   // [T*k]
    const int32_t* active_experts;
    const int32_t* compact_offset;
    const int32_t* compact_ids;
    const WsHeader* hdr;
    uint16_t* act_out;           // gate_up output [P][I]
    float* pair_out;             // down output [P][H] (indexed by pair id)
    int kc;                      // K-chunk staged in shared memory
    int max_tasks;
};
constexpr int kGemvThreads = 256;
constexpr int kGemvMP = 8;       // pairs per pass
constexpr int kGemvRows = 4;     // weight rows per warp
int gemv_smem_bytes(int kc);
cudaError_t launch_gemv(const GemvArgs& args, int grid, cudaStream_t stream, bool pdl);
cudaError_t init_gemv_attributes();
int gemv_blocks_per_sm(int smem_bytes);

// --------------------------------------------------------------- reduce ----
struct ReduceArgs {
    int T, k, H, E, L;
    const float* pair_out;       // [P][H]
    const int32_t* topk_ids;
    const int32_t* lora_ids;
    uint16_t* out;               // [T][H]
};
cudaError_t launch_reduce(const ReduceArgs& args, int grid, cudaStream_t stream, bool pdl);

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
