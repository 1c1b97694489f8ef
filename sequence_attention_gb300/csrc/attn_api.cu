// ABI entry points of the attention step: argument validation and dispatch
// to the fp32 CUDA-core kernel or the tcgen05 tensor-core kernel.
#include <math.h>
#include <string.h>

#include "attn_common.cuh"

namespace ditsp {
namespace {

bool stride_ok(int64_t s, int elem_bytes) { return s >= 0 && ((s * elem_bytes) % 16) == 0; }

// With one output base for every query block (o.stride_q == 0), the blocks'
// output rows [q_row0 + o_row0, + q_len) must not overlap.
bool block_rows_disjoint(const AttnArgs& a) {
    for (int r = 0; r < a.n_q; ++r)
        for (int s = r + 1; s < a.n_q; ++s) {
            if (a.q_len[r] == 0 || a.q_len[s] == 0) continue;
            const long long r0 = (long long)a.q_row0[r] + a.o_row0[r], s0 = (long long)a.q_row0[s] + a.o_row0[s];
            if (r0 < s0 + a.q_len[s] && s0 < r0 + a.q_len[r]) return false;
        }
    return true;
}

dit_status validate_and_launch(AttnArgs& a, const char* who, cudaStream_t st) {
    if (a.B < 1 || a.H < 1 || a.D < 1) return fail(DIT_ERR_INVALID_ARG, "%s: need B, H, D >= 1", who);
    if (!(a.scale > 0.f) || !isfinite(a.scale))
        return fail(DIT_ERR_INVALID_ARG, "%s: scale must be positive and finite", who);
    if (a.n_q < 1 || a.n_q > DIT_MAX_R || a.n_kv < 1 || a.n_kv > DIT_MAX_R)
        return fail(DIT_ERR_INVALID_ARG, "%s: need 1 <= n_q, n_kv <= %d", who, DIT_MAX_R);
    for (int r = 0; r < a.n_q; ++r)
        if (a.q_len[r] < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative query length", who);
    for (int r = 0; r < a.n_kv; ++r)
        if (a.kv_len[r] < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative key length", who);
    if (!dtype_ok(a.qk_dt) || !dtype_ok(a.v_dt) || !dtype_ok(a.o_dt))
        return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    const bool f32 = a.qk_dt == DIT_F32;
    if (f32) {
        if (a.v_dt != DIT_F32 || a.o_dt != DIT_F32)
            return fail(DIT_ERR_UNSUPPORTED, "%s: fp32 Q/K need fp32 V and fp32 O", who);
        if (a.D != 16 && a.D != 32 && a.D != 64 && a.D != 128)
            return fail(DIT_ERR_UNSUPPORTED, "%s: fp32 path supports D in {16,32,64,128}", who);
    } else {
        if (a.v_dt == DIT_F32) return fail(DIT_ERR_UNSUPPORTED, "%s: 16-bit Q/K need 16-bit V", who);
        if (a.D != 64 && a.D != 128)
            return fail(DIT_ERR_UNSUPPORTED, "%s: tensor-core path supports D in {64,128}", who);
    }
    const int qb = dtype_bytes(a.qk_dt), vb = dtype_bytes(a.v_dt), ob = dtype_bytes(a.o_dt);
    const bool ok = stride_ok(a.q.stride_q, qb) && stride_ok(a.q.stride_b, qb) && stride_ok(a.q.stride_s, qb) &&
                    stride_ok(a.q.stride_h, qb) && stride_ok(a.k.stride_kv, qb) && stride_ok(a.k.stride_b, qb) &&
                    stride_ok(a.k.stride_s, qb) && stride_ok(a.k.stride_h, qb) && stride_ok(a.v.stride_kv, vb) &&
                    stride_ok(a.v.stride_b, vb) && stride_ok(a.v.stride_s, vb) && stride_ok(a.v.stride_h, vb) &&
                    stride_ok(a.o.stride_q, ob) && stride_ok(a.o.stride_kv, ob) && stride_ok(a.o.stride_b, ob) &&
                    stride_ok(a.o.stride_s, ob) && stride_ok(a.o.stride_h, ob);
    if (!ok) return fail(DIT_ERR_INVALID_ARG, "%s: strides must be non-negative 16-byte multiples", who);
    // no two results may share an output address (the tensor-core path
    // stores whole row tiles with TMA): a zero output stride is allowed only
    // on a dimension with a single index
    int maxq = 0;
    for (int r = 0; r < a.n_q; ++r) maxq = a.q_len[r] > maxq ? a.q_len[r] : maxq;
    const bool alias = (a.H > 1 && a.o.stride_h == 0) || (maxq > 1 && a.o.stride_s == 0) ||
                       (a.B > 1 && a.o.stride_b == 0) ||
                       (!a.diag && a.n_q > 1 && a.o.stride_q == 0 && !block_rows_disjoint(a)) ||
                       (!a.diag && !a.fold && a.n_kv > 1 && a.o.stride_kv == 0);
    if (alias) return fail(DIT_ERR_INVALID_ARG, "%s: output view maps two results to one address", who);
    // No query rows: nothing is read or written, so the (empty) buffers may
    // be NULL, as an allocator gives for zero bytes.
    if (maxq == 0) return DIT_OK;
    if (!a.q.ptr || !a.o.ptr) return fail(DIT_ERR_INVALID_ARG, "%s: NULL tensor pointer", who);
    if (!aligned16(a.q.ptr) || !aligned16(a.o.ptr))
        return fail(DIT_ERR_INVALID_ARG, "%s: tensor pointers must be 16-byte aligned", who);
    if (a.lse.ptr && (reinterpret_cast<uintptr_t>(a.lse.ptr) & 3))
        return fail(DIT_ERR_INVALID_ARG, "%s: lse pointer misaligned", who);
    bool any_keys = false;
    for (int j = 0; j < a.n_kv; ++j) any_keys |= a.kv_len[j] > 0;
    if (!any_keys && (!a.k.ptr || !a.v.ptr)) {
        // Every key block is empty (O = 0, lse = -inf): K and V are never
        // read, and may be NULL.  The kernels still take descriptors of
        // them, so they get Q's view, which is valid and never used.
        a.k = a.q;
        a.v = a.q;
    }
    if (!a.k.ptr || !a.v.ptr) return fail(DIT_ERR_INVALID_ARG, "%s: NULL tensor pointer", who);
    if (!aligned16(a.k.ptr) || !aligned16(a.v.ptr))
        return fail(DIT_ERR_INVALID_ARG, "%s: tensor pointers must be 16-byte aligned", who);
    if (!a.status) a.status = default_status_word();
    if (!a.status) return fail(DIT_ERR_CUDA, "%s: no device status word", who);
    return f32 ? launch_attn_f32(a, st) : launch_attn_tc(a, st);
}

}  // namespace
}  // namespace ditsp

using namespace ditsp;

extern "C" dit_status dit_attn_partial(int B, int H, int D, float scale, int n_q, const int* q_len, int n_kv,
                                       const int* kv_len, dit_view q, dit_dtype qk_dt, dit_view k, dit_view v,
                                       dit_dtype v_dt, dit_view o, dit_dtype o_dt, dit_lse_view lse,
                                       int* d_status, void* stream) {
    NvtxRange nvtx_range("dit_attn_partial");
    if (!q_len || !kv_len) return fail(DIT_ERR_INVALID_ARG, "dit_attn_partial: NULL length array");
    if (n_q < 1 || n_q > DIT_MAX_R || n_kv < 1 || n_kv > DIT_MAX_R)
        return fail(DIT_ERR_INVALID_ARG, "dit_attn_partial: need 1 <= n_q, n_kv <= %d", DIT_MAX_R);
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.B = B; a.H = H; a.D = D; a.n_q = n_q; a.n_kv = n_kv; a.scale = scale;
    for (int r = 0; r < n_q; ++r) a.q_len[r] = q_len[r];
    for (int r = 0; r < n_kv; ++r) a.kv_len[r] = kv_len[r];
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.qk_dt = qk_dt; a.v_dt = v_dt; a.o_dt = o_dt; a.lse = lse; a.status = d_status;
    return validate_and_launch(a, "dit_attn_partial", (cudaStream_t)stream);
}

extern "C" dit_status dit_attn_ring(int B, int H, int D, float scale, int n_q, const int* q_len, int n_kv,
                                    const int* kv_len, dit_view q, dit_dtype qk_dt, dit_view k, dit_view v,
                                    dit_dtype v_dt, dit_view o, dit_dtype o_dt, dit_lse_view lse, int* d_status,
                                    void* stream) {
    NvtxRange nvtx_range("dit_attn_ring");
    if (!q_len || !kv_len) return fail(DIT_ERR_INVALID_ARG, "dit_attn_ring: NULL length array");
    if (n_q < 1 || n_q > DIT_MAX_R || n_kv < 1 || n_kv > DIT_MAX_R)
        return fail(DIT_ERR_INVALID_ARG, "dit_attn_ring: need 1 <= n_q, n_kv <= %d", DIT_MAX_R);
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.B = B; a.H = H; a.D = D; a.n_q = n_q; a.n_kv = n_kv; a.scale = scale; a.fold = 1;
    for (int r = 0; r < n_q; ++r) a.q_len[r] = q_len[r];
    for (int r = 0; r < n_kv; ++r) a.kv_len[r] = kv_len[r];
    o.stride_kv = 0;                  // one result per query block
    lse.stride_kv = 0;
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.qk_dt = qk_dt; a.v_dt = v_dt; a.o_dt = o_dt; a.lse = lse; a.status = d_status;
    return validate_and_launch(a, "dit_attn_ring", (cudaStream_t)stream);
}

extern "C" dit_status dit_attn_ring_rows(int B, int H, int D, float scale, int n_q, const int* q_len,
                                         const int* o_row0, int n_kv, const int* kv_len, dit_view q, dit_dtype qk_dt,
                                         dit_view k, dit_view v, dit_dtype v_dt, dit_view o, dit_dtype o_dt,
                                         dit_lse_view lse, int* d_status, void* stream) {
    NvtxRange nvtx_range("dit_attn_ring_rows");
    const char* who = "dit_attn_ring_rows";
    if (!q_len || !kv_len || !o_row0) return fail(DIT_ERR_INVALID_ARG, "%s: NULL length or row array", who);
    if (n_q < 1 || n_q > DIT_MAX_R || n_kv < 1 || n_kv > DIT_MAX_R)
        return fail(DIT_ERR_INVALID_ARG, "%s: need 1 <= n_q, n_kv <= %d", who, DIT_MAX_R);
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.B = B; a.H = H; a.D = D; a.n_q = n_q; a.n_kv = n_kv; a.scale = scale; a.fold = 1;
    for (int r = 0; r < n_q; ++r) {
        if (o_row0[r] < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative output row", who);
        a.q_len[r] = q_len[r];
        a.o_row0[r] = o_row0[r];
    }
    for (int r = 0; r < n_kv; ++r) a.kv_len[r] = kv_len[r];
    o.stride_kv = 0;                  // one result per query block
    lse.stride_kv = 0;
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.qk_dt = qk_dt; a.v_dt = v_dt; a.o_dt = o_dt; a.lse = lse; a.status = d_status;
    return validate_and_launch(a, who, (cudaStream_t)stream);
}

extern "C" dit_status dit_attention(int B, int H, int D, float scale, int Sq, int Sk, dit_view q, dit_dtype qk_dt,
                                    dit_view k, dit_view v, dit_dtype v_dt, dit_view o, dit_dtype o_dt,
                                    dit_lse_view lse, int* d_status, void* stream) {
    NvtxRange nvtx_range("dit_attention");
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.B = B; a.H = H; a.D = D; a.n_q = 1; a.n_kv = 1; a.scale = scale;
    a.q_len[0] = Sq; a.kv_len[0] = Sk;
    q.stride_q = q.stride_kv = 0;
    k.stride_q = k.stride_kv = 0;
    v.stride_q = v.stride_kv = 0;
    o.stride_q = o.stride_kv = 0;
    lse.stride_q = lse.stride_kv = 0;
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.qk_dt = qk_dt; a.v_dt = v_dt; a.o_dt = o_dt; a.lse = lse; a.status = d_status;
    return validate_and_launch(a, "dit_attention", (cudaStream_t)stream);
}

extern "C" dit_status dit_attn_varlen(int H, int D, float scale, int nseq, const int* cu_q, const int* cu_k,
                                      dit_view q, dit_dtype qk_dt, dit_view k, dit_view v, dit_dtype v_dt,
                                      dit_view o, dit_dtype o_dt, dit_lse_view lse, int* d_status, void* stream) {
    NvtxRange nvtx_range("dit_attn_varlen");
    const char* who = "dit_attn_varlen";
    if (nseq < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative sequence count", who);
    if (nseq == 0) return DIT_OK;
    if (!cu_q || !cu_k) return fail(DIT_ERR_INVALID_ARG, "%s: NULL offset array", who);
    if (cu_q[0] < 0 || cu_k[0] < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative offset", who);
    for (int s = 0; s < nseq; ++s)
        if (cu_q[s + 1] < cu_q[s] || cu_k[s + 1] < cu_k[s])
            return fail(DIT_ERR_INVALID_ARG, "%s: offsets must not decrease", who);
    // packed rows: no batch or block strides
    q.stride_q = q.stride_kv = q.stride_b = 0;
    k.stride_q = k.stride_kv = k.stride_b = 0;
    v.stride_q = v.stride_kv = v.stride_b = 0;
    o.stride_q = o.stride_kv = o.stride_b = 0;
    lse.stride_q = lse.stride_kv = lse.stride_b = 0;
    // up to DIT_MAX_R sequences per launch, each its own (diagonal) block
    for (int s0 = 0; s0 < nseq; s0 += DIT_MAX_R) {
        const int n = nseq - s0 < DIT_MAX_R ? nseq - s0 : DIT_MAX_R;
        AttnArgs a;
        memset(&a, 0, sizeof(a));
        a.B = 1; a.H = H; a.D = D; a.n_q = n; a.n_kv = n; a.scale = scale; a.diag = 1;
        for (int i = 0; i < n; ++i) {
            a.q_row0[i] = cu_q[s0 + i];
            a.kv_row0[i] = cu_k[s0 + i];
            a.q_len[i] = cu_q[s0 + i + 1] - cu_q[s0 + i];
            a.kv_len[i] = cu_k[s0 + i + 1] - cu_k[s0 + i];
        }
        a.q = q; a.k = k; a.v = v; a.o = o;
        a.qk_dt = qk_dt; a.v_dt = v_dt; a.o_dt = o_dt; a.lse = lse; a.status = d_status;
        const dit_status st = validate_and_launch(a, who, (cudaStream_t)stream);
        if (st != DIT_OK) return st;
    }
    return DIT_OK;
}
