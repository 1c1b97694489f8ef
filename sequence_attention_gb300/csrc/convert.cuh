// Conversion of 8 elements held in registers between the element types of
// the library, with the optional rotary embedding of interleaved pairs;
// shared by the permutation kernels (ulysses.cu, direct.cu).
#pragma once

#include "common.cuh"

namespace ditsp {
namespace {

__device__ __forceinline__ bool narrowing(dit_dtype s, dit_dtype d) {
    return (s == DIT_F32 && d != DIT_F32) || (s == DIT_BF16 && d == DIT_F16);
}

// Convert 8 elements held in registers (SB bytes each) to the destination
// encoding (DB bytes each); narrowing rounds to nearest even.  With `check`,
// a finite value that becomes infinite sets `overflow`.
// True when one of 8 finite values becomes infinite on rounding to the
// 16-bit type t (see overflows16).  The common case -- the largest magnitude
// below the threshold -- costs one max tree and one compare.
__device__ __forceinline__ bool overflows16x8(const float (&f)[8], dit_dtype t) {
    const float lim = t == DIT_F16 ? 65520.f : __uint_as_float(0x7F7F8000u);
    const float m = fmaxf(fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))),
                          fmaxf(fmaxf(fabsf(f[4]), fabsf(f[5])), fmaxf(fabsf(f[6]), fabsf(f[7]))));
    if (m < lim) return false;    // NaN-free maximum below the threshold (a NaN max falls through)
    bool o = false;
#pragma unroll
    for (int e = 0; e < 8; ++e) o |= overflows16(f[e], t);
    return o;
}

template <int SB, int DB>
__device__ __forceinline__ void convert8(const uint4 (&in)[SB / 2], dit_dtype sdt, dit_dtype ddt, bool check,
                                         uint4 (&out)[DB / 2], bool& overflow) {
    if (sdt == ddt) {
#pragma unroll
        for (int h = 0; h < DB / 2; ++h) out[h] = in[h < SB / 2 ? h : 0];
        return;
    }
    Vec8 v;
    load8(&in[0], sdt, v);
    if constexpr (DB == 4) {
        out[0] = make_uint4(__float_as_uint(v.f[0]), __float_as_uint(v.f[1]), __float_as_uint(v.f[2]),
                            __float_as_uint(v.f[3]));
        out[1] = make_uint4(__float_as_uint(v.f[4]), __float_as_uint(v.f[5]), __float_as_uint(v.f[6]),
                            __float_as_uint(v.f[7]));
    } else {
        out[0] = make_uint4(pack2(v.f[0], v.f[1], ddt), pack2(v.f[2], v.f[3], ddt),
                            pack2(v.f[4], v.f[5], ddt), pack2(v.f[6], v.f[7], ddt));
        if (check) overflow |= overflows16x8(v.f, ddt);
    }
}

// Rotate the four interleaved pairs held in 8 elements by the angles with
// cosines c and sines s, in fp32, then convert to the destination type.
template <int SB, int DB>
__device__ __forceinline__ void rope8(const uint4 (&in)[SB / 2], dit_dtype sdt, dit_dtype ddt, float4 c, float4 s,
                                      bool check, uint4 (&out)[DB / 2], bool& overflow) {
    Vec8 v;
    load8(&in[0], sdt, v);
    const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
    Vec8 y;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float x0 = v.f[2 * k], x1 = v.f[2 * k + 1];
        y.f[2 * k] = fmaf(x0, cc[k], -(x1 * ss[k]));
        y.f[2 * k + 1] = fmaf(x0, ss[k], x1 * cc[k]);
    }
    if constexpr (DB == 4) {
        out[0] = make_uint4(__float_as_uint(y.f[0]), __float_as_uint(y.f[1]), __float_as_uint(y.f[2]),
                            __float_as_uint(y.f[3]));
        out[1] = make_uint4(__float_as_uint(y.f[4]), __float_as_uint(y.f[5]), __float_as_uint(y.f[6]),
                            __float_as_uint(y.f[7]));
    } else {
        out[0] = make_uint4(pack2(y.f[0], y.f[1], ddt), pack2(y.f[2], y.f[3], ddt),
                            pack2(y.f[4], y.f[5], ddt), pack2(y.f[6], y.f[7], ddt));
        if (check) overflow |= overflows16x8(y.f, ddt);
    }
}

// 16-byte asynchronous copy global -> shared (no registers held meanwhile).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

}  // namespace
}  // namespace ditsp
