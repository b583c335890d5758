// Device-side helpers shared by the kernels of libmoe.so.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void record_error(uint32_t *err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 16 bytes of elements <-> fp32 registers. VEC = elements per 16 bytes.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int n = 4;
    __device__ __forceinline__ static void load(const float *p, float *v) {
        float4 q = *reinterpret_cast<const float4 *>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    __device__ __forceinline__ static void store(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *v) {
        uint4 q = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Programmatic dependent launch. The forward's kernels are launched with programmatic
// stream serialisation (launch_pdl): a kernel may be scheduled while its predecessor
// on the stream is still running, overlapping its launch and its prologue (barrier
// setup, TMEM allocation) with the predecessor's last wave. pdl_wait() returns once
// the predecessor grid has completed and its memory is visible; every such kernel
// calls it before its first access to global memory, so the chain stays ordered
// (each kernel's predecessor waited for its own predecessor before finishing).
// pdl_launch_dependents() lets the next kernel be scheduled once every CTA of this
// one has issued it; it is issued after pdl_wait(), so a waiting dependent never
// holds an SM that a not yet started CTA of this grid needs. Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_launch_dependents();
}

// Set for the duration of a call whose config carries MOE_DEBUG_NO_PDL: launch_pdl
// then launches plainly (every kernel waits for its predecessor's completion).
extern thread_local bool g_no_pdl;

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_no_pdl ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// SiLU(z) = z / (1 + exp(-z)), fp32, with the fast division intrinsic (within 2 ulp;
// the result is rounded to bf16, or compared at 1e-4 on the fp32 path). The IEEE
// division made the epilogue of the pair kernel's transposed tail tiles slow enough to
// stall the MMAs (Mixtral-shaped product 1 1.46-1.50 vs 1.28-1.31 ms).
__device__ __forceinline__ float silu_f32(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace moe
