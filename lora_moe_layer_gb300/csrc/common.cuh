// common.cuh -- device helpers shared by the libmoelora kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moelora {

// Device status bits, OR-ed into WsHeader::status.
constexpr int kStatusBadExpert = 1;
constexpr int kStatusBadLora = 2;

// First 256 bytes of every workspace.
struct WsHeader {
    int32_t status;           // OR of kStatus* bits seen by the last align/forward
    int32_t num_post_padded;  // padded bucket total
    int32_t n_valid;          // valid pairs (= rows of the compact order)
    int32_t n_active;         // experts with at least one valid pair
    int32_t n_lora_buckets;   // (expert, adapter >= 0) buckets with at least one pair
    int32_t n_shrink_tasks;   // entries of the LoRA shrink task list
    int32_t reserved[58];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte block");

constexpr unsigned kFull = 0xffffffffu;

// --- bf16 bits -> fp32 (exact) --------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf_one(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN kept quiet)
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// fp32 -> bf16 bits by the hardware conversion (round to nearest even; the
// same bits as f32_to_bf16_rne for finite inputs, one instruction)
__device__ __forceinline__ uint16_t f32_to_bf16_cvt(float f) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}

// 8 bf16 (one 16-byte chunk) dotted with 8 fp32, accumulated into acc
__device__ __forceinline__ float dot8(const uint4 w, const float* v, float acc) {
    acc = fmaf(bf_lo(w.x), v[0], acc);
    acc = fmaf(bf_hi(w.x), v[1], acc);
    acc = fmaf(bf_lo(w.y), v[2], acc);
    acc = fmaf(bf_hi(w.y), v[3], acc);
    acc = fmaf(bf_lo(w.z), v[4], acc);
    acc = fmaf(bf_hi(w.z), v[5], acc);
    acc = fmaf(bf_lo(w.w), v[6], acc);
    acc = fmaf(bf_hi(w.w), v[7], acc);
    return acc;
}

__device__ __forceinline__ void unpack8(const uint4 w, float* v) {
    v[0] = bf_lo(w.x); v[1] = bf_hi(w.x);
    v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    v[4] = bf_lo(w.z); v[5] = bf_hi(w.z);
    v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
}

// --- global loads ------------------------------------------------------------
// Streaming read-only 16-byte load that does not allocate in L1 (weights are
// read once per forward).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Read-only 16-byte load through the non-coherent path (inputs of this launch).
__device__ __forceinline__ uint4 ld_ro16(const void* p) {
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// --- programmatic dependent launch --------------------------------------------
// Block until every grid this one depends on has completed and its memory is
// visible.  A no-op when the launch carried no programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to start launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// --- warp reductions ---------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Reduce-scatter of N values across the 32 lanes (N a power of two, 1..32).
// On return v[0] of lane `lane` holds the warp-wide sum of value index
// lane / (32 / N) (each total is replicated on 32 / N adjacent lanes).
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
    int n = N;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const int half = n >> 1;
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; i++) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(kFull, send, o);
                }
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], o);
        }
    }
    return v[0];
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moelora
