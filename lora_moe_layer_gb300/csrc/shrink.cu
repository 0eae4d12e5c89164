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
// For wide buckets (tens of rows) a second kernel below stages A in shared
// memory per CTA instead.  The gate_up launch of either also copies x rows
// into bucket order (the B operand of the gate_up GEMM), so the forward needs
// no separate gather launch.
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

// x rows into bucket order (the gate_up GEMM's B operand), four copies in
// flight per thread, grid-strided over all CTAs of the launch
__device__ void gather_rows(const ShrinkArgs& a) {
    const int K = a.K;
    const int c8 = K >> 3;
    const long total = (long)a.hdr->n_valid * c8;
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i0 = (long)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
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

// z rows of one (bucket, output group) completed by the last split: the S
// partials added in split order, loads in batches of 8
__device__ __forceinline__ void finish_split(const ShrinkArgs& a, int row0, int row1, int col0, int ncol, int tid,
                                             int nthreads) {
    const int r = a.r, S = a.S;
    const int n = (row1 - row0) * ncol;
    for (int idx = tid; idx < n; idx += nthreads) {
        const size_t off = (size_t)(row0 + idx / ncol) * r + col0 + idx % ncol;
        float v = 0.f;
        for (int s0 = 0; s0 < S; s0 += 8) {
            float part[8];
#pragma unroll
            for (int u = 0; u < 8; u++) part[u] = s0 + u < S ? __ldcg(a.z + (size_t)(s0 + u) * a.P * r + off) : 0.f;
#pragma unroll
            for (int u = 0; u < 8; u++)
                if (s0 + u < S) v += part[u];
        }
        a.zfinal[off] = v;
    }
}

__global__ void __launch_bounds__(kThreads, 2) k_shrink(ShrinkArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int L1 = a.L + 1;
    const int r = a.r;
    const int K = a.K;

    if (a.xc) gather_rows(a);

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
                finish_split(a, row0, row1, g * 8, 8, lane, 32);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Wide buckets (prefill: tens of rows per (expert, adapter)): one CTA per
// (bucket, K-split of kSlabK elements) stages the r x kSlabK slab of A[l][e]
// in shared memory once (eight 16-byte loads in flight per thread), and its
// eight warps share the bucket's rows: per row, lanes side by side along K,
// every A row read from shared memory, then a reduce-scatter.  Split-K
// partials are finished by the last CTA of the bucket, in split order.
constexpr int kSlabK = 512;

template <int RP>  // rank rounded up to a power of two (8, 16, 32, 64)
__global__ void __launch_bounds__(kThreads) k_shrink_slab(ShrinkArgs a) {
    extern __shared__ __align__(16) uint16_t slab[];  // [RP][kSlabK]
    __shared__ int s_last;
    pdl_wait();
    pdl_trigger();
    if (a.xc) gather_rows(a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L1 = a.L + 1;
    const int r = a.r, K = a.K, S = a.S;
    const int n_items = a.hdr->n_lora_buckets * S;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int bi = item / S, s = item % S;
        const int b = a.lora_buckets[bi];
        const int e = b / L1, l = b % L1 - 1;
        const int row0 = a.compact_offset[b], row1 = a.compact_offset[b + 1];
        const int k0 = s * kSlabK;
        const int kc = min(kSlabK, K - k0);
        const int chunks = kc >> 3;
        const uint16_t* abase = a.A + ((size_t)(l * a.E + e) * r) * K + k0;

        __syncthreads();  // the previous item's slab is no longer read
        const int n16 = r * chunks;
        for (int c0 = threadIdx.x; c0 < n16; c0 += 8 * kThreads) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int c = c0 + u * kThreads;
                if (c < n16) v[u] = ld_stream16(abase + (size_t)(c / chunks) * K + (c % chunks) * 8);
            }
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int c = c0 + u * kThreads;
                if (c < n16) *reinterpret_cast<uint4*>(slab + (c / chunks) * kSlabK + (c % chunks) * 8) = v[u];
            }
        }
        __syncthreads();

        for (int row = row0 + warp; row < row1; row += kWarps) {
            const uint16_t* in = (a.in_is_x ? a.in + (size_t)(a.compact_ids[row] / a.k) * K : a.in + (size_t)row * K) + k0;
            uint4 xin[kSlabK / 256];
#pragma unroll
            for (int u = 0; u < kSlabK / 256; u++) {
                const int c = lane + 32 * u;
                xin[u] = make_uint4(0, 0, 0, 0);
                if (c < chunks) xin[u] = a.in_is_x ? ld_ro16(in + c * 8) : ld_cg16(in + c * 8);
            }
            float acc[RP];
#pragma unroll
            for (int i = 0; i < RP; i++) acc[i] = 0.f;
#pragma unroll
            for (int u = 0; u < kSlabK / 256; u++) {
                const int c = lane + 32 * u;
                if (c < chunks) {
                    float xv[8];
                    unpack8(xin[u], xv);
#pragma unroll
                    for (int rr = 0; rr < RP; rr++)
                        if (rr < r) acc[rr] = dot8(*reinterpret_cast<const uint4*>(slab + rr * kSlabK + c * 8), xv, acc[rr]);
                }
            }
            float* dst = (S == 1 ? a.zfinal : a.z + (size_t)s * a.P * r) + (size_t)row * r;
            if constexpr (RP <= 32) {
                const float tot = warp_reduce_scatter<RP>(acc, lane);
                const int idx = lane / (32 / RP);
                if (lane % (32 / RP) == 0 && idx < r) dst[idx] = tot;
            } else {
                float lo[32], hi[32];
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    lo[i] = acc[i];
                    hi[i] = acc[32 + i];
                }
                const float tlo = warp_reduce_scatter<32>(lo, lane);
                const float thi = warp_reduce_scatter<32>(hi, lane);
                if (lane < r) dst[lane] = tlo;
                if (32 + lane < r) dst[32 + lane] = thi;
            }
        }

        if (S > 1) {
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[bi], 1) == S - 1;
            __syncthreads();
            if (s_last) {
                __threadfence();
                finish_split(a, row0, row1, 0, r, threadIdx.x, kThreads);
            }
        }
    }
}

template <int RP>
cudaError_t slab_attr() {
    return cudaFuncSetAttribute(k_shrink_slab<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, RP * kSlabK * 2);
}

}  // namespace

cudaError_t init_shrink_attributes() {
    cudaError_t e;
    if ((e = slab_attr<8>()) != cudaSuccess) return e;
    if ((e = slab_attr<16>()) != cudaSuccess) return e;
    if ((e = slab_attr<32>()) != cudaSuccess) return e;
    return slab_attr<64>();
}

int shrink_slab_splits(int K) { return (K + kSlabK - 1) / kSlabK; }

cudaError_t launch_shrink_slab(const ShrinkArgs& args, int grid, cudaStream_t stream, bool pdl) {
    const dim3 g(grid), b(kThreads);
    if (args.r <= 8) return launch_k(k_shrink_slab<8>, g, b, 8 * kSlabK * 2, stream, pdl, args);
    if (args.r <= 16) return launch_k(k_shrink_slab<16>, g, b, 16 * kSlabK * 2, stream, pdl, args);
    if (args.r <= 32) return launch_k(k_shrink_slab<32>, g, b, 32 * kSlabK * 2, stream, pdl, args);
    return launch_k(k_shrink_slab<64>, g, b, 64 * kSlabK * 2, stream, pdl, args);
}

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
