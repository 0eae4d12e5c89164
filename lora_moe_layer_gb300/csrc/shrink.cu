// shrink.cu -- LoRA shrink z = A[l][e] . in for every adapter pair, as a
// skinny GEMM split over warps.
//
// The blog ("Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Kernel optimizations")
// notes that the shrink has only r outputs (tens) per row against a reduction
// over h_in (thousands), so one thread group per output leaves the GPU idle;
// it splits the K sum across groups and adds the partial sums.  Here the unit
// of work is one warp: an item is (bucket (e, l >= 0), group of 8 of the r
// outputs, K-split).  The warp streams its 8 rows of A[l][e] over its K range
// with 16-byte loads (lanes side by side along K, two 256-element steps in
// flight) against each row of the bucket (x for gate_up, act for down), keeps
// 8 accumulators per bucket row, and finishes with a shuffle reduce-scatter.  Without a
// K-split the warp writes z directly; with one, it writes its partial and the
// warp that completes an item's last split (a per-item arrival counter decides)
// adds the partials in split order, so the result is deterministic.  No shared
// memory and no block-wide barrier: warps run independently.
//
// The gate_up launch also copies x rows into bucket order (the B operand of
// the gate_up GEMM), so the forward needs no separate gather launch.
#include "common.cuh"
#include "kernels.cuh"

namespace moelora {

namespace {

// L2-only 16-byte load for rows an earlier kernel of the chain wrote
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRB = 1;  // bucket rows per pass

__global__ void __launch_bounds__(kThreads, 2) k_shrink(ShrinkArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int L1 = a.L + 1;
    const int r = a.r;
    const int K = a.K;

    if (a.xc) {
        // x rows into bucket order, four copies in flight per thread
        const int c8 = K >> 3;
        const long total = (long)a.hdr->n_valid * c8;
        const long stride = (long)gridDim.x * kThreads;
        for (long i0 = (long)blockIdx.x * kThreads + threadIdx.x; i0 < total; i0 += 4 * stride) {
            uint4 v[4];
            long dst[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const long idx = i0 + u * stride;
                dst[u] = -1;
                if (idx < total) {
                    const int q = (int)(idx / c8), c = (int)(idx % c8);
                    dst[u] = (long)q * K + c * 8;
                    v[u] = ld_ro16(a.in + (size_t)(a.compact_ids[q] / a.k) * K + c * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (dst[u] >= 0) *reinterpret_cast<uint4*>(a.xc + dst[u]) = v[u];
        }
    }

    const int groups = r >> 3;
    const int S = a.S;
    const int ks = a.ks;  // K elements per split, a multiple of 256
    const long n_items = (long)a.hdr->n_lora_buckets * groups * S;
    for (long item = (long)blockIdx.x * kWarps + (threadIdx.x >> 5); item < n_items;
         item += (long)gridDim.x * kWarps) {
        const int s = (int)(item % S);
        const long bg = item / S;               // (bucket, group) index
        const int g = (int)(bg % groups);
        const int bi = (int)(bg / groups);
        const int b = a.lora_buckets[bi];
        const int e = b / L1, l = b % L1 - 1;
        const int row0 = a.compact_offset[b], row1 = a.compact_offset[b + 1];
        const int k0 = s * ks, k1 = min(K, k0 + ks);
        const uint16_t* arow = a.A + (((size_t)l * a.E + e) * r + g * 8) * K;

        for (int rb = row0; rb < row1; rb += kRB) {
            const uint16_t* in[kRB];
            bool rok[kRB];
#pragma unroll
            for (int i = 0; i < kRB; i++) {
                rok[i] = rb + i < row1;
                const int row = rok[i] ? rb + i : rb;
                in[i] = a.in_is_x ? a.in + (size_t)(a.compact_ids[row] / a.k) * K : a.in + (size_t)row * K;
            }
            float acc[kRB][8];
#pragma unroll
            for (int i = 0; i < kRB; i++)
#pragma unroll
                for (int j = 0; j < 8; j++) acc[i][j] = 0.f;

            for (int kk = k0 + lane * 8; kk < k1; kk += 512) {
                // two 256-element steps: 8 rows of A and the bucket rows, all loads issued first
                uint4 w0[8], w1[8], x0[kRB], x1[kRB];
                const bool two = kk + 256 < k1;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    w0[j] = ld_stream16(arow + (size_t)j * K + kk);
                    w1[j] = two ? ld_stream16(arow + (size_t)j * K + kk + 256) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < kRB; i++) {
                    x0[i] = x1[i] = make_uint4(0, 0, 0, 0);
                    if (rok[i]) {
                        x0[i] = a.in_is_x ? ld_ro16(in[i] + kk) : ld_cg16(in[i] + kk);
                        if (two) x1[i] = a.in_is_x ? ld_ro16(in[i] + kk + 256) : ld_cg16(in[i] + kk + 256);
                    }
                }
#pragma unroll
                for (int i = 0; i < kRB; i++) {
                    float xv[8];
                    unpack8(x0[i], xv);
#pragma unroll
                    for (int j = 0; j < 8; j++) acc[i][j] = dot8(w0[j], xv, acc[i][j]);
                    unpack8(x1[i], xv);
#pragma unroll
                    for (int j = 0; j < 8; j++) acc[i][j] = dot8(w1[j], xv, acc[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < kRB; i++) {
                // lane 4m holds output m of the group after the reduce-scatter
                const float v = warp_reduce_scatter<8>(acc[i], lane);
                if (rok[i] && (lane & 3) == 0) {
                    float* dst = S == 1 ? a.zfinal : a.z + (size_t)s * a.P * r;
                    dst[(size_t)(rb + i) * r + g * 8 + (lane >> 2)] = v;
                }
            }
        }

        if (S > 1) {
            // split-K completion: the last split of this (bucket, group) adds them up
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = atomicAdd(&a.counters[bg], 1) == S - 1;
            last = __shfl_sync(kFull, last, 0);
            if (last) {
                __threadfence();
                const int n = (row1 - row0) * 8;
                for (int idx = lane; idx < n; idx += 32) {
                    const size_t off = (size_t)(row0 + idx / 8) * r + g * 8 + (idx & 7);
                    float v = 0.f;
                    for (int s0 = 0; s0 < S; s0 += 8) {  // loads in batches of 8, sums in split order
                        float part[8];
#pragma unroll
                        for (int u = 0; u < 8; u++)
                            part[u] = s0 + u < S ? __ldcg(a.z + (size_t)(s0 + u) * a.P * r + off) : 0.f;
#pragma unroll
                        for (int u = 0; u < 8; u++)
                            if (s0 + u < S) v += part[u];
                    }
                    a.zfinal[off] = v;
                }
            }
        }
    }
}

}  // namespace

int shrink_splits(int K, long items_no_split) {
    // about 2048 warps in flight (a GB300 holds ~9700), in K slices of 256 or more
    const long want = 2048;
    long s = items_no_split > 0 ? (want + items_no_split - 1) / items_no_split : 1;
    const long max_s = (K + 255) / 256;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    return (int)s;
}

int shrink_split_len(int K, int S) {
    const int per = (K + S - 1) / S;
    return (per + 255) / 256 * 256;
}

cudaError_t launch_shrink(const ShrinkArgs& args, int grid, cudaStream_t stream, bool pdl) {
    return launch_k(k_shrink, dim3(grid), dim3(kThreads), 0, stream, pdl, args);
}

int shrink_warps_per_block() { return kWarps; }

}  // namespace moelora
