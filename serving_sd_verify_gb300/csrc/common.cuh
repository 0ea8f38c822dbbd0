// Device helpers shared by the kernel files of libsdverify.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace sdv {

// exact widening of a bf16 bit pattern
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// 8 bf16 values packed in a 16-byte word -> 8 floats
__device__ __forceinline__ void unpack_bf16x8(const uint4 w, float (&f)[8]) {
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xffff0000u);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;   // elements per 16-byte load
    __device__ __forceinline__ static float load(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static void load_vec(const float *p, float (&f)[4]) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static float load(const __nv_bfloat16 *p) {
        return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short *>(p)));
    }
    __device__ __forceinline__ static void load_vec(const __nv_bfloat16 *p, float (&f)[8]) {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        unpack_bf16x8(v, f);
    }
};

// streaming 16-byte load that does not allocate in L1 (read-once data)
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void set_fault(unsigned int *fault, unsigned int bits) {
    if (fault) atomicOr(fault, bits);
}

// (value, index) pair ordering of the argmax: larger value wins; equal values
// go to the lower index.  NaN never wins against an ordered value.
__device__ __forceinline__ bool argmax_better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

}  // namespace sdv
