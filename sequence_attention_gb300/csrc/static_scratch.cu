// dit_attn_ring_merge_static: the ring's partial attention followed by the
// log-sum-exp merge, with the partials kept in a fixed device array that the
// library owns instead of in caller memory.  The entry point allocates
// nothing; it exists for callers that cannot call cudaMalloc.
#include <string.h>

#include <atomic>

#include "common.cuh"

namespace ditsp {
namespace {

// The partials and their log-sum-exp rows of one call.  Part of the
// library's device code: a device holds it from the time the library's code
// is loaded there until the process exits.
static __device__ __align__(256) unsigned char g_ring_scratch[DIT_RING_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<unsigned char*> g_scratch_addr[kMaxDevices];

// Device address of g_ring_scratch on the current device, looked up once per
// device (the name is a host-side stand-in, not an address a kernel can use).
dit_status scratch_address(unsigned char** out, const char* who) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(DIT_ERR_UNSUPPORTED, "%s: device index %d", who, dev);
    unsigned char* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress((void**)&p, g_ring_scratch);
        if (e != cudaSuccess || !p)
            return fail(DIT_ERR_CUDA, "%s: cudaGetSymbolAddress of the scratch array: %s", who,
                        cudaGetErrorString(e));
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return DIT_OK;
}

}  // namespace
}  // namespace ditsp

using namespace ditsp;

extern "C" dit_status dit_attn_ring_merge_static(int B, int H, int D, float scale, int n_q, const int* q_len, int n_kv,
                                                 const int* kv_len, dit_view q, dit_dtype qk_dt, dit_view k,
                                                 dit_view v, dit_dtype v_dt, dit_view o, dit_dtype o_dt,
                                                 dit_lse_view lse, int* d_status, void* stream) {
    NvtxRange nvtx_range("dit_attn_ring_merge_static");
    const char* who = "dit_attn_ring_merge_static";
    // Everything that needs no device is checked first, so a request that
    // does not fit is refused without touching CUDA.
    if (!q_len || !kv_len) return fail(DIT_ERR_INVALID_ARG, "%s: NULL length array", who);
    if (n_q < 1 || n_q > DIT_MAX_R || n_kv < 1 || n_kv > DIT_MAX_R)
        return fail(DIT_ERR_INVALID_ARG, "%s: need 1 <= n_q, n_kv <= %d", who, DIT_MAX_R);
    if (B < 1 || H < 1 || D < 1) return fail(DIT_ERR_INVALID_ARG, "%s: need B, H, D >= 1", who);
    int maxq = 0;
    for (int r = 0; r < n_q; ++r) {
        if (q_len[r] < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative query length", who);
        maxq = q_len[r] > maxq ? q_len[r] : maxq;
    }
    // No query rows: dit_attn_ring checks the other arguments and launches
    // nothing (its buffers may be NULL).
    if (maxq == 0)
        return dit_attn_ring(B, H, D, scale, n_q, q_len, n_kv, kv_len, q, qk_dt, k, v, v_dt, o, o_dt, lse, d_status,
                             stream);
    // fp32 partials [n_q][n_kv][B][maxq][H][D], then fp32 lse rows
    // [n_q][n_kv][B][H][maxq] from the next 256-byte boundary.  The size is
    // built factor by factor against the limit, so no product can wrap.
    const unsigned long long cap = DIT_RING_STATIC_SCRATCH_BYTES;
    const unsigned long long factors[6] = {(unsigned long long)n_q, (unsigned long long)n_kv, (unsigned long long)B,
                                           (unsigned long long)H, (unsigned long long)maxq, 4ull * (unsigned long long)D};
    unsigned long long part_bytes = 1;
    bool fits = true;
    for (int f = 0; f < 6 && fits; ++f) {
        fits = part_bytes <= cap / factors[f];
        part_bytes *= fits ? factors[f] : 1ull;
    }
    const unsigned long long rows = fits ? part_bytes / factors[5] : 0;
    const unsigned long long lse_off = (part_bytes + 255ull) & ~255ull;
    if (!fits || lse_off + rows * 4ull > cap)
        return fail(DIT_ERR_INVALID_ARG,
                    "%s: the partials of %d x %d blocks, B=%d, H=%d, %d rows, D=%d do not fit the library's fixed "
                    "scratch of %llu bytes (use dit_attn_partial + dit_attn_merge_lse with caller buffers, or "
                    "dit_attn_ring)",
                    who, n_q, n_kv, B, H, maxq, D, cap);

    unsigned char* base = nullptr;
    dit_status s = scratch_address(&base, who);
    if (s != DIT_OK) return s;

    const int64_t sh = D, ss = (int64_t)H * D, sb = (int64_t)maxq * H * D;
    dit_view parts;
    memset(&parts, 0, sizeof(parts));
    parts.ptr = base;
    parts.stride_h = sh;
    parts.stride_s = ss;
    parts.stride_b = sb;
    parts.stride_kv = sb * B;
    parts.stride_q = sb * B * n_kv;
    dit_lse_view lse_parts;
    memset(&lse_parts, 0, sizeof(lse_parts));
    lse_parts.ptr = reinterpret_cast<float*>(base + lse_off);
    lse_parts.stride_h = maxq;
    lse_parts.stride_b = (int64_t)H * maxq;
    lse_parts.stride_kv = (int64_t)B * H * maxq;
    lse_parts.stride_q = (int64_t)n_kv * B * H * maxq;

    s = dit_attn_partial(B, H, D, scale, n_q, q_len, n_kv, kv_len, q, qk_dt, k, v, v_dt, parts, DIT_F32, lse_parts,
                         d_status, stream);
    if (s != DIT_OK) return s;
    return dit_attn_merge_lse(B, H, D, n_q, q_len, n_kv, parts, DIT_F32, lse_parts, o, o_dt, lse, stream);
}
