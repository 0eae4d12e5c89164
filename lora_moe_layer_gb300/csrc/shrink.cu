// shrink.cu -- LoRA shrink z = A[l][e] . in as a split-K skinny GEMM.
//
// The blog ("Efficiently serve dozens of fine-tuned models with vLLM ...",
// section "Kernel optimizations") notes that the shrink has only r outputs
// (tens) per row against a reduction over h_in (thousands), so giving each
// output to one thread group leaves the GPU idle; it splits the K sum over
// many groups and combines the partial sums.  The same split here: one work
// item is (bucket (e, l >= 0), K-split s); it stages the r x KC slab of
// A[l][e] in shared memory once (coalesced 16-byte loads), then every warp
// takes rows of the bucket, each lane holding 8 consecutive K elements per
// 256-element step, and a shuffle reduce-scatter leaves one output per lane.
// Each split writes its partials to z[s][row][:]; the CTA that completes a
// bucket's last split (an arrival counter per bucket decides which) sums the S
// partials in split order into zfinal[row][:].  The order of the sum is fixed,
// so the result is deterministic; only the choice of the summing CTA varies.
#include "common.cuh"
#include "kernels.cuh"

namespace moelora {

namespace {

constexpr int kShrinkThreads = 256;
constexpr int kShrinkWarps = kShrinkThreads / 32;

template <int RP>  // rank padded to a power of two (8, 16, 32, 64)
__global__ void __launch_bounds__(kShrinkThreads) k_shrink(ShrinkArgs a) {
    extern __shared__ __align__(16) uint16_t a_slab[];  // [RP][kShrinkKC]
    pdl_wait();
    pdl_trigger();
    __shared__ int s_last;
    const int n_items = a.hdr->n_lora_buckets * a.S;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L1 = a.L + 1;
    const int r = a.r;

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int bi = item / a.S, s = item % a.S;
        const int b = a.lora_buckets[bi];
        const int e = b / L1, l = b % L1 - 1;
        const int row0 = a.compact_offset[b], row1 = a.compact_offset[b + 1];
        const int k0 = s * kShrinkKC;
        const int kc = min(kShrinkKC, a.K - k0);  // multiple of 8
        const int chunks = kc >> 3;               // 16-byte chunks per A row in this split

        __syncthreads();  // previous item's slab fully consumed
        const uint16_t* Abase = a.A + ((size_t)(l * a.E + e) * r) * a.K + k0;
        for (int c = threadIdx.x; c < r * chunks; c += kShrinkThreads) {
            const int rr = c / chunks, cc = c % chunks;
            *reinterpret_cast<uint4*>(a_slab + rr * kShrinkKC + cc * 8) =
                ld_stream16(Abase + (size_t)rr * a.K + cc * 8);
        }
        __syncthreads();

        for (int row = row0 + warp; row < row1; row += kShrinkWarps) {
            const uint16_t* in_row = a.in_is_x
                ? a.in + (size_t)(a.compact_ids[row] / a.k) * a.K + k0
                : a.in + (size_t)row * a.K + k0;
            float acc[RP];
#pragma unroll
            for (int i = 0; i < RP; i++) acc[i] = 0.f;
            for (int c = lane; c < chunks; c += 32) {
                float xv[8];
                unpack8(ld_ro16(in_row + c * 8), xv);
#pragma unroll
                for (int rr = 0; rr < RP; rr++) {
                    if (rr < r) {
                        const uint4 w = *reinterpret_cast<const uint4*>(a_slab + rr * kShrinkKC + c * 8);
                        acc[rr] = dot8(w, xv, acc[rr]);
                    }
                }
            }
            float* zrow = a.z + ((size_t)s * a.P + row) * r;
            if constexpr (RP <= 32) {
                const float tot = warp_reduce_scatter<RP>(acc, lane);
                const int idx = lane / (32 / RP);
                if (lane % (32 / RP) == 0 && idx < r) zrow[idx] = tot;
            } else {
                float lo[32], hi[32];
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    lo[i] = acc[i];
                    hi[i] = acc[32 + i];
                }
                const float tlo = warp_reduce_scatter<32>(lo, lane);
                const float thi = warp_reduce_scatter<32>(hi, lane);
                if (lane < r) zrow[lane] = tlo;
                if (32 + lane < r) zrow[32 + lane] = thi;
            }
        }

        // split-K completion: the last split of this bucket to finish sums them all
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[bi], 1) == a.S - 1;
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int n = (row1 - row0) * r;
            for (int idx = threadIdx.x; idx < n; idx += kShrinkThreads) {
                const size_t off = (size_t)row0 * r + idx;
                float v = 0.f;
                for (int s2 = 0; s2 < a.S; s2++) v += __ldcg(a.z + (size_t)s2 * a.P * r + off);
                a.zfinal[off] = v;
            }
        }
    }
}

template <int RP>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(k_shrink<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                RP * kShrinkKC * 2);
}

}  // namespace

cudaError_t init_shrink_attributes() {
    cudaError_t e;
    if ((e = set_attr<8>()) != cudaSuccess) return e;
    if ((e = set_attr<16>()) != cudaSuccess) return e;
    if ((e = set_attr<32>()) != cudaSuccess) return e;
    return set_attr<64>();
}

int shrink_blocks_per_sm() { return 4; }

cudaError_t launch_shrink(const ShrinkArgs& args, int grid, cudaStream_t stream, bool pdl) {
    const dim3 block(kShrinkThreads);
    if (args.r <= 8)
        return launch_k(k_shrink<8>, dim3(grid), block, 8 * kShrinkKC * 2, stream, pdl, args);
    if (args.r <= 16)
        return launch_k(k_shrink<16>, dim3(grid), block, 16 * kShrinkKC * 2, stream, pdl, args);
    if (args.r <= 32)
        return launch_k(k_shrink<32>, dim3(grid), block, 32 * kShrinkKC * 2, stream, pdl, args);
    return launch_k(k_shrink<64>, dim3(grid), block, 64 * kShrinkKC * 2, stream, pdl, args);
}

}  // namespace moelora
