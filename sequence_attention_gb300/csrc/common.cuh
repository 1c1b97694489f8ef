// Shared host/device helpers of libditsp: error reporting, element types,
// vectorised 8-element load/convert/store.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "ditsp.h"

#include <nvtx3/nvToolsExt.h>

namespace ditsp {

// NVTX range around one ABI call: names the call on a profiler timeline
// (Nsight Systems); without a tool attached each push/pop is a no-op.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---- host-side error reporting (thread-local message) ----------------------
dit_status fail(dit_status s, const char* fmt, ...);
dit_status check_launch(const char* what);
int* default_status_word();      // device address of the library status word
int num_sms();                   // SM count of the current device (cached)

inline bool dtype_ok(dit_dtype t) { return t == DIT_F32 || t == DIT_BF16 || t == DIT_F16; }
// element types plus the record-encoded e4m3 type, valid only on the wire
inline bool wire_ok(dit_dtype t) { return dtype_ok(t) || t == DIT_E4M3; }
__host__ __device__ inline int dtype_bytes(dit_dtype t) { return t == DIT_F32 ? 4 : 2; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- programmatic dependent launch -------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization allowed: it may begin while the previous kernel in the
// stream drains.  A kernel runs its input-independent prologue, then
// pdl_wait() (which returns once every earlier kernel has completed and its
// writes are visible) before it reads or writes any tensor, and calls
// pdl_trigger() when its CTA has finished its work.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- device-side element access --------------------------------------------
// Eight consecutive elements of one type, moved as 16-byte (16-bit types) or
// 2x16-byte (float) vectors.  Callers guarantee 16-byte alignment.

struct Vec8 {
    float f[8];
};

__device__ __forceinline__ void load8(const void* p, dit_dtype t, Vec8& v) {
    if (t == DIT_F32) {
        const float4* q = reinterpret_cast<const float4*>(p);
        float4 a = q[0], b = q[1];
        v.f[0] = a.x; v.f[1] = a.y; v.f[2] = a.z; v.f[3] = a.w;
        v.f[4] = b.x; v.f[5] = b.y; v.f[6] = b.z; v.f[7] = b.w;
    } else {
        uint4 r = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (t == DIT_BF16) {
                __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
                float2 f = __bfloat1622float2(h);
                v.f[2 * i] = f.x; v.f[2 * i + 1] = f.y;
            } else {
                __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
                float2 f = __half22float2(h);
                v.f[2 * i] = f.x; v.f[2 * i + 1] = f.y;
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, dit_dtype t) {
    if (t == DIT_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void store8(void* p, dit_dtype t, const Vec8& v) {
    if (t == DIT_F32) {
        float4* q = reinterpret_cast<float4*>(p);
        q[0] = make_float4(v.f[0], v.f[1], v.f[2], v.f[3]);
        q[1] = make_float4(v.f[4], v.f[5], v.f[6], v.f[7]);
    } else {
        uint4 r;
        r.x = pack2(v.f[0], v.f[1], t);
        r.y = pack2(v.f[2], v.f[3], t);
        r.z = pack2(v.f[4], v.f[5], t);
        r.w = pack2(v.f[6], v.f[7], t);
        *reinterpret_cast<uint4*>(p) = r;
    }
}

// True when a finite x becomes infinite on rounding to nearest even into the
// 16-bit type t: |x| at or above the midpoint between t's largest finite
// value and the next power of two (65520 for f16, (2 - 2^-8) * 2^127 for
// bf16), where the tie goes to the even neighbour, infinity.
__device__ __forceinline__ bool overflows16(float x, dit_dtype t) {
    const float lim = t == DIT_F16 ? 65520.f : __uint_as_float(0x7F7F8000u);
    return fabsf(x) >= lim && !isinf(x);
}

__device__ __forceinline__ void store8_zero(void* p, dit_dtype t) {
    uint4 z = make_uint4(0, 0, 0, 0);
    uint4* q = reinterpret_cast<uint4*>(p);
    q[0] = z;
    if (t == DIT_F32) q[1] = z;
}

// Raw copy of 8 elements of the same type (bit-exact, NaN payloads kept).
__device__ __forceinline__ void copy8(void* dst, const void* src, dit_dtype t) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = s[0];
    if (t == DIT_F32) d[1] = s[1];
}

// Unsigned division by a divisor fixed at launch, as a multiply-high and a
// shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with s = ceil(log2 d) and m = floor(2^32 (2^s - d)
// / d) + 1, n / d = (mulhi(n, m) + n) >> s for every n < 2^31.
struct FastDiv {
    uint32_t d, m, s;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.s = 0;
    while ((1ull << f.s) < d) ++f.s;
    f.m = (uint32_t)(((1ull << 32) * ((1ull << f.s) - d)) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
    return (uint32_t)(((unsigned long long)__umulhi(n, f.m) + n) >> f.s);
}

}  // namespace ditsp
