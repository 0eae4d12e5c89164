// reduce.cu -- top-k weighted aggregation:
//   out[t] = bf16(sum_j sum_s pair_out[s][t*k + j]).
//
// The router's k experts of a token are aggregated ("Efficiently serve dozens
// of fine-tuned models with vLLM ...", section "Implementing multi-LoRA
// inference for MoE models in vLLM"); the down kernel has already applied the
// top-k weights.  When the down GEMM splits K, each split s wrote its own
// fp32 slab, and the slabs are added here; without a split the per-pair
// outputs come in bf16 (the activation type).  Both sums run in fp32 in a
// fixed order (slot j = 0 .. k-1, inside it split s = 0 .. nsplit-1:
// deterministic), then one round-to-nearest-even to bf16.  Pairs that carry
// an out-of-range id were left out upstream and are skipped here.  Four hidden
// elements per thread: 16-byte fp32 or 8-byte bf16 loads, 8-byte bf16 stores.
#include "common.cuh"
#include "kernels.cuh"

namespace moelora {

namespace {

__device__ __forceinline__ void add4(float4& s, const float4& v) {
    s.x += v.x;
    s.y += v.y;
    s.z += v.z;
    s.w += v.w;
}

template <bool SPLIT>
__global__ void __launch_bounds__(256) k_reduce(ReduceArgs a) {
    pdl_wait();
    pdl_trigger();
    const int H4 = a.H >> 2;
    const long n = (long)a.T * H4;
    const size_t split4 = a.split_stride / 4;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
        const int t = (int)(idx / H4), h4 = (int)(idx % H4);
        const int l = a.lora_ids[t];
        const bool l_ok = l >= -1 && l < a.L;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        // every slot's row is loaded (rows of left-out pairs exist but are not
        // added), so the k loads go out together
#pragma unroll 4
        for (int j = 0; j < a.k; j++) {
            const int p = t * a.k + j;
            const int e = a.topk_ids[p];
            const float4* src = reinterpret_cast<const float4*>(a.pair_out + (size_t)p * a.H) + h4;
            float4 v = __ldcs(src);
            if (SPLIT) {
                float4 u[kMaxSplitSlabs - 1];
#pragma unroll
                for (int sp = 1; sp < kMaxSplitSlabs; sp++)
                    if (sp < a.nsplit) u[sp - 1] = __ldcs(src + sp * split4);
#pragma unroll
                for (int sp = 1; sp < kMaxSplitSlabs; sp++)
                    if (sp < a.nsplit) add4(v, u[sp - 1]);
            }
            if (l_ok && e >= 0 && e < a.E) add4(s, v);
        }
        uint2 o;
        o.x = (uint32_t)f32_to_bf16_rne(s.x) | ((uint32_t)f32_to_bf16_rne(s.y) << 16);
        o.y = (uint32_t)f32_to_bf16_rne(s.z) | ((uint32_t)f32_to_bf16_rne(s.w) << 16);
        reinterpret_cast<uint2*>(a.out + (size_t)t * a.H)[h4] = o;
    }
}

// The same sum over bf16 per-pair outputs (no K split): eight hidden elements
// per thread, one 16-byte load per slot, four slots' loads in flight before
// their adds (in slot order)
__global__ void __launch_bounds__(256) k_reduce_bf16(ReduceArgs a) {
    pdl_wait();
    pdl_trigger();
    const int H8 = a.H >> 3;
    const long n = (long)a.T * H8;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
        const int t = (int)(idx / H8), h8 = (int)(idx % H8);
        const int l = a.lora_ids[t];
        const bool l_ok = l >= -1 && l < a.L;
        float s[8];
#pragma unroll
        for (int i = 0; i < 8; i++) s[i] = 0.f;
        for (int j0 = 0; j0 < a.k; j0 += 4) {
            uint4 w[4];
            bool use[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                use[q] = false;
                if (j0 + q < a.k) {
                    const int p = t * a.k + j0 + q;
                    const int e = a.topk_ids[p];
                    use[q] = l_ok && e >= 0 && e < a.E;
                    w[q] = __ldcs(reinterpret_cast<const uint4*>(a.pair_out16 + (size_t)p * a.H) + h8);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; q++) {
                if (use[q]) {
                    s[0] += bf_lo(w[q].x); s[1] += bf_hi(w[q].x);
                    s[2] += bf_lo(w[q].y); s[3] += bf_hi(w[q].y);
                    s[4] += bf_lo(w[q].z); s[5] += bf_hi(w[q].z);
                    s[6] += bf_lo(w[q].w); s[7] += bf_hi(w[q].w);
                }
            }
        }
        uint4 o;
        o.x = (uint32_t)f32_to_bf16_rne(s[0]) | ((uint32_t)f32_to_bf16_rne(s[1]) << 16);
        o.y = (uint32_t)f32_to_bf16_rne(s[2]) | ((uint32_t)f32_to_bf16_rne(s[3]) << 16);
        o.z = (uint32_t)f32_to_bf16_rne(s[4]) | ((uint32_t)f32_to_bf16_rne(s[5]) << 16);
        o.w = (uint32_t)f32_to_bf16_rne(s[6]) | ((uint32_t)f32_to_bf16_rne(s[7]) << 16);
        reinterpret_cast<uint4*>(a.out + (size_t)t * a.H)[h8] = o;
    }
}

}  // namespace

cudaError_t launch_reduce(const ReduceArgs& args, int grid, cudaStream_t stream, bool pdl) {
    if (args.nsplit < 1 || args.nsplit > kMaxSplitSlabs) return cudaErrorInvalidValue;
    if (args.nsplit > 1) {
        if (!args.pair_out) return cudaErrorInvalidValue;
        return launch_k(k_reduce<true>, dim3(grid), dim3(256), 0, stream, pdl, args);
    }
    if (args.pair_out16) return launch_k(k_reduce_bf16, dim3(grid), dim3(256), 0, stream, pdl, args);
    if (!args.pair_out) return cudaErrorInvalidValue;
    return launch_k(k_reduce<false>, dim3(grid), dim3(256), 0, stream, pdl, args);
}

}  // namespace moelora
