// The Ulysses all-to-all as permutation kernels over virtual ranks that live
// in one GPU's memory (edge-dit.cpp "Parallel execution": packed QKV send
// path, receive preparation, head-to-sequence path; SGLang Diffusion
// "Parallelism Overview", The Ulysses transport: an all-to-all is a
// permutation, so a copy in one memory is bit-identical to any transport).
//
// Every buffer in the exchange is a sequence of "runs": Hl*D contiguous
// elements = the Hl heads of one rank's head group for one (plane, batch,
// row).  A run is contiguous on both sides of every step, so each kernel
// moves whole runs with 16-byte vectors: one warp per run, lanes over
// 8-element chunks.  Two wire orders exist:
//   A (sequence side): rank (r,u)'s buffer = for v: [planes][B][L_u] runs
//      index  np*B*U*off_u + v*np*B*L_u + (p*B+b)*L_u + i
//   B (head side):     rank (r,v)'s buffer = for u: [planes][B][L_u] runs
//      index  np*B*U*off_r + v*np*B*S_r + np*B*(off_u-off_r) + (p*B+b)*L_u + i
// Seq-to-head: pack writes A, the exchange copies A->B, unpack reads B.
// Head-to-seq: pack writes B, the exchange copies B->A, unpack reads A.
#include <string.h>

#include "common.cuh"

namespace ditsp {
namespace {

enum Mode { PACK_S2H = 0, UNPACK_H2S, PACK_H2S, UNPACK_S2H, A2A_S2H, A2A_H2S };

struct RunArgs {
    dit_sp_layout L;
    int np;
    const void* src[3];
    void* dst[3];
    dit_dtype src_dt[3];
    dit_dtype dst_dt[3];
    int* range_flag;
    long long nruns;
};

struct Run {
    int r, u, v, p, b, i;
};

__device__ __forceinline__ int rank_of_row(const dit_sp_layout& L, int t) {
    int lo = 0, hi = L.U * L.R - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (L.rank_off[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int ring_of_row(const dit_sp_layout& L, int t) {
    int r = 0;
    for (int k = 1; k < L.R; ++k)
        if (L.ring_off[k] <= t && L.ring_len[k] > 0) r = k;
    return r;
}

__device__ __forceinline__ Run decode_A(const dit_sp_layout& L, int np, long long a) {
    const long long per_row = (long long)np * L.B * L.U;
    const int rid = rank_of_row(L, (int)(a / per_row));
    Run x;
    x.r = rid / L.U; x.u = rid % L.U;
    const long long Lu = L.rank_len[rid];
    long long local = a - per_row * L.rank_off[rid];
    const long long blk = (long long)np * L.B * Lu;
    x.v = (int)(local / blk);
    long long rem = local - x.v * blk;
    const int pb = (int)(rem / Lu);
    x.i = (int)(rem - pb * Lu);
    x.p = pb / L.B; x.b = pb % L.B;
    return x;
}

__device__ __forceinline__ Run decode_B(const dit_sp_layout& L, int np, long long bi) {
    const long long per_row = (long long)np * L.B * L.U;
    Run x;
    x.r = ring_of_row(L, (int)(bi / per_row));
    const int offr = L.ring_off[x.r];
    const long long Sr = L.ring_len[x.r];
    long long local = bi - per_row * offr;
    const long long grp = (long long)np * L.B * Sr;
    x.v = (int)(local / grp);
    long long rem = local - x.v * grp;
    const int rid = rank_of_row(L, offr + (int)(rem / ((long long)np * L.B)));
    x.u = rid - x.r * L.U;
    const long long Lu = L.rank_len[rid];
    rem -= (long long)np * L.B * (L.rank_off[rid] - offr);
    const int pb = (int)(rem / Lu);
    x.i = (int)(rem - pb * Lu);
    x.p = pb / L.B; x.b = pb % L.B;
    return x;
}

__device__ __forceinline__ long long index_A(const dit_sp_layout& L, int np, const Run& x) {
    const int rid = x.r * L.U + x.u;
    const long long Lu = L.rank_len[rid];
    return (long long)np * L.B * L.U * L.rank_off[rid] + (long long)x.v * np * L.B * Lu +
           ((long long)x.p * L.B + x.b) * Lu + x.i;
}

__device__ __forceinline__ long long index_B(const dit_sp_layout& L, int np, const Run& x) {
    const int rid = x.r * L.U + x.u;
    const int offr = L.ring_off[x.r];
    return (long long)np * L.B * L.U * offr + (long long)x.v * np * L.B * L.ring_len[x.r] +
           (long long)np * L.B * (L.rank_off[rid] - offr) +
           ((long long)x.p * L.B + x.b) * L.rank_len[rid] + x.i;
}

// element offset of the run's first head in a seq-layout plane [B][S][H][D]
// (only meaningful when the group has a real head)
__device__ __forceinline__ long long seq_offset(const dit_sp_layout& L, const Run& x) {
    const int row = L.rank_off[x.r * L.U + x.u] + x.i;
    return (((long long)x.b * L.S + row) * L.H + (long long)x.v * L.Hl) * L.D;
}

// element offset in a head-layout plane [R][B][S_cap][Hp][D]
__device__ __forceinline__ long long head_offset(const dit_sp_layout& L, const Run& x) {
    const int row = L.rank_off[x.r * L.U + x.u] - L.ring_off[x.r] + x.i;
    return ((((long long)x.r * L.B + x.b) * L.S_cap + row) * L.Hp + (long long)x.v * L.Hl) * L.D;
}

__device__ __forceinline__ bool narrowing(dit_dtype s, dit_dtype d) {
    return (s == DIT_F32 && d != DIT_F32) || (s == DIT_BF16 && d == DIT_F16);
}

template <int MODE>
__global__ void __launch_bounds__(256, 4) run_kernel(const __grid_constant__ RunArgs A) {
    const dit_sp_layout& L = A.L;
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int run_elems = L.Hl * L.D;
    const int nch = run_elems >> 3;
    bool overflow = false;

    for (long long ri = warp0; ri < A.nruns; ri += nwarps) {
        Run x;
        if (MODE == PACK_S2H || MODE == UNPACK_H2S || MODE == A2A_H2S) x = decode_A(L, A.np, ri);
        else x = decode_B(L, A.np, ri);
        const int p = x.p;
        // real heads of this head group; heads at or past nreal are padding
        const int nreal = min(max(L.H - x.v * L.Hl, 0), L.Hl);

        const char* src;
        char* dst;
        dit_dtype sdt, ddt;
        int src_heads = L.Hl;   // source heads that hold data (rest read as 0)
        int dst_heads = L.Hl;   // destination heads that are written
        long long so = 0, doff = 0;
        if (MODE == PACK_S2H) {
            sdt = A.src_dt[p]; ddt = A.dst_dt[0];
            so = nreal > 0 ? seq_offset(L, x) : 0; doff = ri * run_elems;
            src = (const char*)A.src[p]; dst = (char*)A.dst[0];
            src_heads = nreal;
        } else if (MODE == UNPACK_H2S) {
            sdt = A.src_dt[0]; ddt = A.dst_dt[0];
            so = ri * run_elems; doff = nreal > 0 ? seq_offset(L, x) : 0;
            src = (const char*)A.src[0]; dst = (char*)A.dst[0];
            dst_heads = nreal;
        } else if (MODE == PACK_H2S) {
            sdt = A.src_dt[0]; ddt = A.dst_dt[0];
            so = head_offset(L, x); doff = ri * run_elems;
            src = (const char*)A.src[0]; dst = (char*)A.dst[0];
            src_heads = nreal;
        } else if (MODE == UNPACK_S2H) {
            sdt = A.src_dt[0]; ddt = A.dst_dt[p];
            so = ri * run_elems; doff = head_offset(L, x);
            src = (const char*)A.src[0]; dst = (char*)A.dst[p];
        } else if (MODE == A2A_S2H) {
            sdt = ddt = A.src_dt[0];
            so = index_A(L, A.np, x) * run_elems; doff = ri * run_elems;
            src = (const char*)A.src[0]; dst = (char*)A.dst[0];
        } else {  // A2A_H2S
            sdt = ddt = A.src_dt[0];
            so = index_B(L, A.np, x) * run_elems; doff = ri * run_elems;
            src = (const char*)A.src[0]; dst = (char*)A.dst[0];
        }
        src += so * dtype_bytes(sdt);
        dst += doff * dtype_bytes(ddt);
        const int sb = 8 * dtype_bytes(sdt), db = 8 * dtype_bytes(ddt);
        const bool same = (sdt == ddt);
        const bool check_range = (MODE == UNPACK_S2H) && A.range_flag && narrowing(sdt, ddt);

        if (same) {
            // bit-exact move: 16 (or 32) bytes per chunk, four chunks in flight
            for (int c0 = lane; c0 < nch; c0 += 128) {
                uint4 raw[4][2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = c0 + 32 * k;
                    raw[k][0] = raw[k][1] = make_uint4(0, 0, 0, 0);
                    if (c < nch && (c * 8) / L.D < src_heads) {
                        const uint4* q = reinterpret_cast<const uint4*>(src + (long long)c * sb);
                        raw[k][0] = q[0];
                        if (sb == 32) raw[k][1] = q[1];
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = c0 + 32 * k;
                    if (c < nch && (c * 8) / L.D < dst_heads) {
                        uint4* q = reinterpret_cast<uint4*>(dst + (long long)c * db);
                        q[0] = raw[k][0];
                        if (db == 32) q[1] = raw[k][1];
                    }
                }
            }
        } else {
            // converting move: through fp32, rounded to nearest even
            for (int c0 = lane; c0 < nch; c0 += 64) {
                Vec8 val[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int c = c0 + 32 * k;
#pragma unroll
                    for (int e = 0; e < 8; ++e) val[k].f[e] = 0.f;
                    if (c < nch && (c * 8) / L.D < src_heads) load8(src + (long long)c * sb, sdt, val[k]);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int c = c0 + 32 * k;
                    if (c < nch && (c * 8) / L.D < dst_heads) {
                        char* d = dst + (long long)c * db;
                        store8(d, ddt, val[k]);
                        if (check_range) {
                            Vec8 back;
                            load8(d, ddt, back);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                overflow |= isinf(back.f[e]) && !isinf(val[k].f[e]);
                        }
                    }
                }
            }
        }
    }
    if (overflow) *A.range_flag = (int)DIT_ERR_RANGE;
}

// Host-side check of a caller-supplied layout: every field must be what
// dit_sp_layout_init would have produced for its (B, S, H, D, U, R).
dit_status check_layout(const dit_sp_layout* L, const char* who) {
    if (!L) return fail(DIT_ERR_INVALID_ARG, "%s: layout is NULL", who);
    dit_sp_layout ref;
    if (dit_sp_layout_init(L->B, L->S, L->H, L->D, L->U, L->R, &ref) != DIT_OK)
        return fail(DIT_ERR_INVALID_ARG, "%s: layout sizes invalid", who);
    bool ok = ref.Hp == L->Hp && ref.Hl == L->Hl && ref.S_cap == L->S_cap;
    for (int r = 0; ok && r < L->R; ++r)
        ok = ref.ring_len[r] == L->ring_len[r] && ref.ring_off[r] == L->ring_off[r];
    for (int i = 0; ok && i < L->R * L->U; ++i)
        ok = ref.rank_len[i] == L->rank_len[i] && ref.rank_off[i] == L->rank_off[i];
    if (!ok) return fail(DIT_ERR_INVALID_ARG, "%s: layout tables are inconsistent", who);
    if (L->D % 8 != 0)
        return fail(DIT_ERR_UNSUPPORTED, "%s: head dim %d is not a multiple of 8", who, L->D);
    return DIT_OK;
}

template <int MODE>
dit_status launch_runs(const RunArgs& a, cudaStream_t st, const char* who) {
    if (a.nruns == 0) return DIT_OK;
    long long blocks = (a.nruns + 7) / 8;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    run_kernel<MODE><<<(unsigned)blocks, 256, 0, st>>>(a);
    return check_launch(who);
}

}  // namespace
}  // namespace ditsp

using namespace ditsp;

extern "C" dit_status dit_ulysses_pack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                       const void* const* src, dit_dtype src_dt, void* send,
                                       dit_dtype wire_dt, void* stream) {
    const char* who = "dit_ulysses_pack";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!dtype_ok(src_dt) || !dtype_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3 || (dir == DIT_HEAD_TO_SEQ && nplanes != 1))
        return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3 (1 for head-to-seq)", who);
    if (!src || !send || !aligned16(send)) return fail(DIT_ERR_INVALID_ARG, "%s: send NULL or misaligned", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    for (int p = 0; p < nplanes; ++p) {
        if (!src[p] || !aligned16(src[p])) return fail(DIT_ERR_INVALID_ARG, "%s: src[%d] NULL or misaligned", who, p);
        a.src[p] = src[p];
        a.src_dt[p] = src_dt;
    }
    a.dst[0] = send;
    a.dst_dt[0] = wire_dt;
    a.nruns = (long long)nplanes * L->B * L->U * L->S;
    cudaStream_t st = (cudaStream_t)stream;
    return dir == DIT_SEQ_TO_HEAD ? launch_runs<PACK_S2H>(a, st, who) : launch_runs<PACK_H2S>(a, st, who);
}

extern "C" dit_status dit_a2a_sim(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                  const void* send, void* recv, dit_dtype wire_dt, void* stream) {
    const char* who = "dit_a2a_sim";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!dtype_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3) return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3", who);
    if (!send || !recv || !aligned16(send) || !aligned16(recv) || send == recv)
        return fail(DIT_ERR_INVALID_ARG, "%s: send/recv NULL, misaligned or identical", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    a.src[0] = send; a.src_dt[0] = wire_dt;
    a.dst[0] = recv; a.dst_dt[0] = wire_dt;
    a.nruns = (long long)nplanes * L->B * L->U * L->S;
    cudaStream_t st = (cudaStream_t)stream;
    return dir == DIT_SEQ_TO_HEAD ? launch_runs<A2A_S2H>(a, st, who) : launch_runs<A2A_H2S>(a, st, who);
}

extern "C" dit_status dit_ulysses_unpack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                         const void* recv, dit_dtype wire_dt, void* const* dst,
                                         const dit_dtype* dst_dt, int* d_range_flag, void* stream) {
    const char* who = "dit_ulysses_unpack";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!dtype_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad wire dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3 || (dir == DIT_HEAD_TO_SEQ && nplanes != 1))
        return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3 (1 for head-to-seq)", who);
    if (!recv || !aligned16(recv) || !dst || !dst_dt)
        return fail(DIT_ERR_INVALID_ARG, "%s: recv/dst NULL or misaligned", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    a.src[0] = recv; a.src_dt[0] = wire_dt;
    for (int p = 0; p < nplanes; ++p) {
        if (!dst[p] || !aligned16(dst[p])) return fail(DIT_ERR_INVALID_ARG, "%s: dst[%d] NULL or misaligned", who, p);
        if (!dtype_ok(dst_dt[p])) return fail(DIT_ERR_INVALID_ARG, "%s: bad dst dtype", who);
        a.dst[p] = dst[p];
        a.dst_dt[p] = dst_dt[p];
    }
    a.range_flag = d_range_flag;
    a.nruns = (long long)nplanes * L->B * L->U * L->S;
    cudaStream_t st = (cudaStream_t)stream;
    return dir == DIT_SEQ_TO_HEAD ? launch_runs<UNPACK_S2H>(a, st, who) : launch_runs<UNPACK_H2S>(a, st, who);
}
