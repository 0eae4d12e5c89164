// gemv.cu -- grouped GEMV for decode-sized expert groups, with the LoRA
// expand fused into the same accumulation and the activation / top-k weight
// in the epilogue.
//
// Layer math ("Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Implementing multi-LoRA
// inference for MoE models in vLLM", Figure 1): per routed pair,
//   gate_up:  g = W1[e] x + B1[l][e] z1,  act = SiLU(g[0:I]) * g[I:2I]
//   down:     d = W2[e] act + B2[l][e] z2, pair_out = w * d
// where z1, z2 are the LoRA shrink outputs (split-K partials summed here in
// fixed order).  The blog fuses the LoRA add into the expand kernel (section
// "Kernel optimizations"); here the expand term is added to the base dot
// product before anything leaves registers.
//
// Work decomposition: a task is (active expert, block of output rows); its
// CTA walks the expert's rows (all of its pairs, any adapter mix) in passes of
// kGemvMP pairs.  Each warp streams kGemvRows weight rows with 16-byte
// non-allocating loads (every weight byte is read from HBM once per pass),
// lane c handling K elements [8c, 8c+8) of every 256-element step; the pairs'
// input rows sit in shared memory.  A 32-way shuffle reduce-scatter then
// leaves lane = (row, pair) holding one finished dot product.  For gate_up a
// warp's four rows are two gate rows and the two matching up rows, so
// SiLU(gate) * up needs only one shuffle.
#include "common.cuh"
#include "kernels.cuh"

namespace moelora {

namespace {

constexpr int kWarps = kGemvThreads / 32;
constexpr int MP = kGemvMP;
constexpr int NR = kGemvRows;
constexpr int kZStride = 64;  // floats per pair in the z staging area (r <= 64)
static_assert(NR * MP == 32, "one (row, pair) result per lane");

__device__ __forceinline__ float silu_f(float u) { return u / (1.0f + expf(-u)); }

template <bool GATE_UP>
__global__ void __launch_bounds__(kGemvThreads, 2) k_gemv(GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                  // [MP][kc]
    float* zs = reinterpret_cast<float*>(smem + (size_t)MP * a.kc * 2); // [MP][kZStride]
    __shared__ int s_pair[MP];
    __shared__ int s_lora[MP];
    __shared__ float s_w[MP];

    pdl_wait();
    pdl_trigger();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L1 = a.L + 1;
    const int N = GATE_UP ? a.I : a.H;          // output units (gate/up row pairs for gate_up)
    const int K = GATE_UP ? a.H : a.I;
    constexpr int kUnitsPerWarp = GATE_UP ? NR / 2 : NR;
    constexpr int kUnitsPerCta = kWarps * kUnitsPerWarp;
    const int nblk = (N + kUnitsPerCta - 1) / kUnitsPerCta;
    const int n_tasks = a.hdr->n_active * nblk;
    const bool has_lora = a.B != nullptr && a.zpart != nullptr;
    const int r = a.r;

    for (int task = blockIdx.x; task < n_tasks; task += gridDim.x) {
        const int ai = task / nblk, blk = task % nblk;
        const int e = a.active_experts[ai];
        const int q0 = a.compact_offset[e * L1], q1 = a.compact_offset[(e + 1) * L1];
        const int u0 = blk * kUnitsPerCta + warp * kUnitsPerWarp;

        // this warp's weight rows
        const uint16_t* wrow[NR];
        bool wok[NR];
#pragma unroll
        for (int j = 0; j < NR; j++) {
            int out_row, unit;
            if (GATE_UP) {
                unit = u0 + (j & 1);
                out_row = (j < 2) ? unit : a.I + unit;
            } else {
                unit = u0 + j;
                out_row = unit;
            }
            wok[j] = unit < N;
            const size_t rows_per_expert = GATE_UP ? 2 * (size_t)a.I : (size_t)a.H;
            wrow[j] = a.W + ((size_t)e * rows_per_expert + (wok[j] ? out_row : 0)) * K;
        }

        for (int pc = q0; pc < q1; pc += MP) {
            const int m = min(MP, q1 - pc);
            __syncthreads();  // previous pass done with s_*, zs, xs
            if (threadIdx.x < MP) {
                const int i = threadIdx.x;
                if (i < m) {
                    const int p = a.compact_ids[pc + i];
                    s_pair[i] = p;
                    s_lora[i] = a.lora_ids[p / a.k];
                    s_w[i] = a.topk_weights[p];
                } else {
                    s_pair[i] = -1;
                    s_lora[i] = -1;
                    s_w[i] = 0.f;
                }
            }
            __syncthreads();
            if (has_lora) {
                // z = sum over the K-splits of the shrink partials, fixed order
                for (int idx = threadIdx.x; idx < MP * r; idx += kGemvThreads) {
                    const int i = idx / r, rr = idx % r;
                    float v = 0.f;
                    if (i < m && s_lora[i] >= 0) {
                        const float* zp = a.zpart + (size_t)(pc + i) * r + rr;
                        for (int s = 0; s < a.S; s++) v += zp[(size_t)s * a.P * r];
                    }
                    zs[i * kZStride + rr] = v;
                }
            }

            float acc[NR][MP];
#pragma unroll
            for (int j = 0; j < NR; j++)
#pragma unroll
                for (int i = 0; i < MP; i++) acc[j][i] = 0.f;

            for (int k0 = 0; k0 < K; k0 += a.kc) {
                const int kcur = min(a.kc, K - k0);
                const int chunks = kcur >> 3;
                __syncthreads();  // xs free
                for (int c = threadIdx.x; c < m * chunks; c += kGemvThreads) {
                    const int i = c / chunks, cc = c % chunks;
                    const uint16_t* src = GATE_UP
                        ? a.in + (size_t)(s_pair[i] / a.k) * a.H + k0 + cc * 8
                        : a.in + (size_t)(pc + i) * a.I + k0 + cc * 8;
                    *reinterpret_cast<uint4*>(xs + (size_t)i * a.kc + cc * 8) = ld_ro16(src);
                }
                __syncthreads();

                // two 256-element steps per iteration: 8 weight loads in flight per lane
                int c = lane;
                for (; c + 32 < chunks; c += 64) {
                    uint4 w0[NR], w1[NR];
#pragma unroll
                    for (int j = 0; j < NR; j++) {
                        w0[j] = wok[j] ? ld_stream16(wrow[j] + k0 + c * 8) : make_uint4(0, 0, 0, 0);
                        w1[j] = wok[j] ? ld_stream16(wrow[j] + k0 + (c + 32) * 8) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int i = 0; i < MP; i++) {
                        if (i < m) {
                            float xv[8];
                            unpack8(*reinterpret_cast<const uint4*>(xs + (size_t)i * a.kc + c * 8), xv);
#pragma unroll
                            for (int j = 0; j < NR; j++) acc[j][i] = dot8(w0[j], xv, acc[j][i]);
                            unpack8(*reinterpret_cast<const uint4*>(xs + (size_t)i * a.kc + (c + 32) * 8), xv);
#pragma unroll
                            for (int j = 0; j < NR; j++) acc[j][i] = dot8(w1[j], xv, acc[j][i]);
                        }
                    }
                }
                if (c < chunks) {
                    uint4 w0[NR];
#pragma unroll
                    for (int j = 0; j < NR; j++)
                        w0[j] = wok[j] ? ld_stream16(wrow[j] + k0 + c * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int i = 0; i < MP; i++) {
                        if (i < m) {
                            float xv[8];
                            unpack8(*reinterpret_cast<const uint4*>(xs + (size_t)i * a.kc + c * 8), xv);
#pragma unroll
                            for (int j = 0; j < NR; j++) acc[j][i] = dot8(w0[j], xv, acc[j][i]);
                        }
                    }
                }
            }

            // lane <- (row j = lane / MP, pair i = lane % MP)
            float v[32];
#pragma unroll
            for (int j = 0; j < NR; j++)
#pragma unroll
                for (int i = 0; i < MP; i++) v[j * MP + i] = acc[j][i];
            float g = warp_reduce_scatter<32>(v, lane);
            const int j = lane / MP, i = lane % MP;
            const int unit = GATE_UP ? u0 + (j & 1) : u0 + j;
            const bool ok = i < m && unit < N;
            const int l = s_lora[i];
            if (has_lora && ok && l >= 0) {
                const int out_row = GATE_UP ? ((j < 2) ? unit : a.I + unit) : unit;
                const size_t rows_per_expert = GATE_UP ? 2 * (size_t)a.I : (size_t)a.H;
                const uint16_t* brow = a.B + (((size_t)l * a.E + e) * rows_per_expert + out_row) * r;
                const float* z = zs + i * kZStride;
                float dlt = 0.f;
                for (int c8 = 0; c8 < r; c8 += 8) {
                    const uint4 bw = ld_ro16(brow + c8);
                    dlt = dot8(bw, z + c8, dlt);
                }
                g += dlt;
            }
            if (GATE_UP) {
                const float up = __shfl_xor_sync(kFull, g, 16);
                if (lane < 16 && ok)
                    a.act_out[(size_t)(pc + i) * a.I + unit] = f32_to_bf16_rne(silu_f(g) * up);
            } else {
                if (ok) a.pair_out[(size_t)s_pair[i] * a.H + unit] = s_w[i] * g;
            }
        }
    }
}

}  // namespace

int gemv_smem_bytes(int kc) { return MP * kc * 2 + MP * kZStride * 4; }

cudaError_t init_gemv_attributes() {
    const int max_smem = gemv_smem_bytes(4096);
    cudaError_t e = cudaFuncSetAttribute(k_gemv<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_gemv<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

int gemv_blocks_per_sm(int smem_bytes) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<true>, kGemvThreads, smem_bytes) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

cudaError_t launch_gemv(const GemvArgs& args, int grid, cudaStream_t stream, bool pdl) {
    const int smem = gemv_smem_bytes(args.kc);
    if (args.gate_up)
        return launch_k(k_gemv<true>, dim3(grid), dim3(kGemvThreads), smem, stream, pdl, args);
    return launch_k(k_gemv<false>, dim3(grid), dim3(kGemvThreads), smem, stream, pdl, args);
}

}  // namespace moelora
