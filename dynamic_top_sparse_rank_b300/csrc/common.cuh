// Device helpers shared by the kernels of libssa.so (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssa.h"

#define SSA_DEVINL __device__ __forceinline__

namespace ssa {

constexpr float kLog2e = 1.4426950408889634f;

// Report a device-side error bit without trapping.
SSA_DEVINL void report(int32_t* dev_status, int bit) {
    if (dev_status) atomicOr(dev_status, bit);
}

// ---- element access ------------------------------------------------------

// Eight bf16 values packed in a uint4 -> eight floats (exact).
SSA_DEVINL void bf16x8_to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

SSA_DEVINL void f32x4_to_f32(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}

// 16 bytes of a row as floats: 8 elements for bf16, 4 for f32.
template <bool BF16>
struct Vec16 {
    static constexpr int E = BF16 ? 8 : 4;
    SSA_DEVINL static void to_f32(const uint4& v, float* f) {
        if constexpr (BF16)
            bf16x8_to_f32(v, f);
        else
            f32x4_to_f32(v, f);
    }
};

SSA_DEVINL uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// Streaming 16-byte load that does not allocate in L1 (data used once per CTA).
SSA_DEVINL uint4 ld_nc_na16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---- ordering keys ---------------------------------------------------------

// Monotone map float -> uint32: a < b  <=>  key(a) < key(b) (for non-NaN).
// -0.0 is folded onto +0.0 first, so equal floats give equal keys.
SSA_DEVINL uint32_t f32_order_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

SSA_DEVINL float order_key_f32(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// Head mapping of the gather attention: H query heads, H_kv key/value heads
// and H_idx index lists (both dividing H); grouped == 0 is the plain layout
// (one of each per head).
struct HeadMap {
    int H, H_kv, H_idx;
    int grouped, head_inner;
};

// Composite selection key: larger score first, then smaller index first.
SSA_DEVINL uint64_t sel_key(uint32_t okey, uint32_t j) {
    return (static_cast<uint64_t>(okey) << 32) | static_cast<uint64_t>(~j);
}
SSA_DEVINL uint32_t sel_key_index(uint64_t key) { return ~static_cast<uint32_t>(key); }
SSA_DEVINL uint32_t sel_key_okey(uint64_t key) { return static_cast<uint32_t>(key >> 32); }

}  // namespace ssa
