// The Ulysses permutation in one pass (edge-dit.cpp "Parallel execution":
// packed QKV send path, receive preparation, head-to-sequence path; SGLang
// Diffusion "Parallelism Overview", The Ulysses transport).
//
// When every virtual rank lives in the same memory, rank v's receive block
// from rank u is rank u's send block to v, so the exchange can alias the two
// (recv[v][u] == send[u][v]) and pack -> exchange -> unpack composes into one
// permutation from the sequence layout straight to the head layout, and back.
// Each element is read once and written once: no send or receive buffer.
// The results are bit-identical to the three-call path with the wire in the
// source type (one rounding, source to destination type).
//
//   seq -> head:  head-layout row (plane p, ring block r, batch b, row i) =
//                 sequence row t = ring_off[r] + i of plane p, batch b, its H
//                 heads followed by Hp - H zero heads; rows t >= S (sequence
//                 padding) are zero.  Optional RoPE of chosen planes.
//   head -> seq:  sequence row (b, t < S) = the first H heads of head-layout
//                 row (r, b, t - ring_off[r]).
//
// Work division: the destination is a flat sequence of 8-element chunks, rows
// of cpr chunks each.  Every warp takes one contiguous equal share of the
// chunks (rounded to whole 32-chunk steps), so all warps of the grid finish
// together; lanes walk the share 32 chunks apart.  Per batch of kItems
// chunks a lane issues every 16-byte load first, then converts and stores.
// The grid holds as many blocks as fit on the SMs at once (or fewer for
// small copies): one wave, no tail.
#include <string.h>

#include "convert.cuh"
#include "sp_index.cuh"

namespace ditsp {
namespace {

constexpr int kDirThreads = 256;
constexpr int kDirItems = 8;     // chunks per lane in flight

struct DirectArgs {
    dit_sp_layout L;
    int np;                      // planes (seq -> head); 1 for head -> seq
    // sequence side: rows [0, split) in seq[p] ([B][split][H][D]) and rows
    // [split, S) in seq2[p] ([B][S - split][H][D]); split == 0: all rows in
    // seq[p] ([B][S][H][D])
    char* seq[3];
    char* seq2[3];
    int split;
    char* head[3];               // head-layout planes [R][B][S_cap][Hp][D]
    dit_dtype src_dt[3], dst_dt[3];
    int* range_flag;
    const float* cos_tab;
    const float* sin_tab;
    unsigned rope_planes;
    long long nrows;             // destination rows
    int cpr;                     // chunks per destination row
    int creal;                   // chunks of a row that carry real heads (H * D / 8)
    long long share;             // chunks per warp
};

// Byte address of the first element of sequence row t of batch b.
__device__ __forceinline__ char* seq_row(const DirectArgs& A, char* const (&s)[3], char* const (&s2)[3], int p,
                                         int b, int t, int eb) {
    const dit_sp_layout& L = A.L;
    long long rows = L.S, row = t;
    char* base = s[p];
    if (A.split > 0) {
        if (t >= A.split) {
            base = s2[p];
            rows = L.S - A.split;
            row = t - A.split;
        } else {
            rows = A.split;
        }
    }
    return base + (((long long)b * rows + row) * L.H) * L.D * eb;
}

__device__ __forceinline__ long long head_row_elems(const dit_sp_layout& L, int b, int t) {
    const int r = ring_of_row(L, t);
    const int i = t - L.ring_off[r];
    return (((long long)r * L.B + b) * L.S_cap + i) * L.Hp * L.D;
}

template <bool S2H, int SB, int DB, bool ROPE>
__global__ void __launch_bounds__(kDirThreads) direct_kernel(const __grid_constant__ DirectArgs A) {
    const dit_sp_layout& L = A.L;
    const int lane = threadIdx.x & 31;
    const long long warp = (long long)blockIdx.x * (kDirThreads / 32) + (threadIdx.x >> 5);
    const long long q0 = warp * A.share;
    const long long q1 = min(A.nrows * A.cpr, q0 + A.share);
    pdl_wait();
    if (q0 >= q1) {
        pdl_trigger();
        return;
    }
    const bool want_check = S2H && A.range_flag != nullptr;
    bool overflow = false;
    // the lane's next chunk: destination row `row`, chunk `c` of it
    long long q = q0 + lane;
    long long row = q / A.cpr;
    int c = (int)(q - row * A.cpr);
    // decoded row (refreshed when `row` changes)
    long long cur = -1;
    const char* srow = nullptr;
    char* drow = nullptr;
    int rp = 0, rt = 0;
    bool rreal = false;
    auto decode = [&]() {
        cur = row;
        if (S2H) {
            const long long per_plane = (long long)L.B * L.S_pad;
            rp = (int)(row / per_plane);
            const long long rem = row - rp * per_plane;
            const int b = (int)(rem / L.S_pad);
            rt = (int)(rem - (long long)b * L.S_pad);
            rreal = rt < L.S;
            drow = A.head[rp] + head_row_elems(L, b, rt) * DB;
            srow = rreal ? seq_row(A, A.seq, A.seq2, rp, b, rt, SB) : nullptr;
        } else {
            const int b = (int)(row / L.S);
            rt = (int)(row - (long long)b * L.S);
            rp = 0;
            rreal = true;
            srow = A.head[0] + head_row_elems(L, b, rt) * SB;
            drow = seq_row(A, A.seq, A.seq2, 0, b, rt, DB);
        }
    };
    constexpr int NI = kDirItems;
    uint4 raw[NI][SB / 2];
    char* dptr[NI];
    int meta[NI];      // plane, | 4 when rotated; -1: no chunk
    long long tab[NI]; // rotary table offset (floats) of the chunk's first pair
    for (long long qb = q0; qb < q1; qb += 32 * NI) {
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            meta[k] = -1;
#pragma unroll
            for (int h = 0; h < SB / 2; ++h) raw[k][h] = make_uint4(0, 0, 0, 0);
            if (q < q1) {
                if (row != cur) decode();
                dptr[k] = drow + (long long)c * 8 * DB;
                int m = rp;
                if (rreal && c < A.creal) {
                    const uint4* s = reinterpret_cast<const uint4*>(srow + (long long)c * 8 * SB);
#pragma unroll
                    for (int h = 0; h < SB / 2; ++h) raw[k][h] = s[h];
                    if (ROPE && ((A.rope_planes >> rp) & 1u)) {
                        m |= 4;
                        tab[k] = (long long)rt * (L.D >> 1) + (((c * 8) % L.D) >> 1);
                    }
                }
                meta[k] = m;
            }
            q += 32;
            c += 32;
            while (c >= A.cpr) {
                c -= A.cpr;
                ++row;
            }
        }
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            if (meta[k] < 0) continue;
            const int p = meta[k] & 3;
            const dit_dtype sdt = A.src_dt[p], ddt = A.dst_dt[p];
            uint4 o[DB / 2];
            if (ROPE && (meta[k] & 4)) {
                const float4 cs = __ldg(reinterpret_cast<const float4*>(A.cos_tab + tab[k]));
                const float4 sn = __ldg(reinterpret_cast<const float4*>(A.sin_tab + tab[k]));
                rope8<SB, DB>(raw[k], sdt, ddt, cs, sn, want_check && ddt != DIT_F32, o, overflow);
            } else {
                convert8<SB, DB>(raw[k], sdt, ddt, want_check && narrowing(sdt, ddt), o, overflow);
            }
            uint4* d = reinterpret_cast<uint4*>(dptr[k]);
#pragma unroll
            for (int h = 0; h < DB / 2; ++h) d[h] = o[h];
        }
    }
    if (overflow) *A.range_flag = (int)DIT_ERR_RANGE;
    pdl_trigger();
}

template <bool S2H, int SB, int DB, bool ROPE>
dit_status launch_direct_sized(DirectArgs& a, cudaStream_t st, const char* who) {
    auto kern = direct_kernel<S2H, SB, DB, ROPE>;
    // blocks resident per SM, looked up once per instantiation
    static const int occ = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDirThreads, 0) != cudaSuccess || n <= 0) n = 2;
        return n;
    }();
    const long long total = a.nrows * a.cpr;
    const long long per_block = (long long)kDirThreads * kDirItems;
    long long blocks = (total + per_block - 1) / per_block;
    const long long resident = (long long)num_sms() * occ;
    if (blocks > resident) blocks = resident;
    const long long warps = blocks * (kDirThreads / 32);
    long long share = (total + warps - 1) / warps;
    share = (share + 31) / 32 * 32;
    a.share = share;
    cudaError_t e = launch_pdl(kern, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

template <bool S2H, bool ROPE>
dit_status launch_direct(DirectArgs& a, cudaStream_t st, const char* who) {
    const int sb = dtype_bytes(a.src_dt[0]), db = dtype_bytes(a.dst_dt[0]);
    for (int p = 1; p < a.np; ++p)
        if (dtype_bytes(a.dst_dt[p]) != db)
            return fail(DIT_ERR_UNSUPPORTED, "%s: planes of one call need destination types of one size", who);
    if (sb == 2 && db == 2) return launch_direct_sized<S2H, 2, 2, ROPE>(a, st, who);
    if (sb == 4 && db == 4) return launch_direct_sized<S2H, 4, 4, ROPE>(a, st, who);
    if (sb == 4 && db == 2) return launch_direct_sized<S2H, 4, 2, ROPE>(a, st, who);
    return launch_direct_sized<S2H, 2, 4, ROPE>(a, st, who);
}

// Checks shared by both directions: the sequence-side pointer pair of
// plane p given split (0: one tensor).
dit_status seq_pair_ok(const void* s, const void* s2, int split, int S, const char* who, int p) {
    if (!s || !aligned16(s)) return fail(DIT_ERR_INVALID_ARG, "%s: sequence tensor %d NULL or misaligned", who, p);
    if (split > 0 && split < S && (!s2 || !aligned16(s2)))
        return fail(DIT_ERR_INVALID_ARG, "%s: second sequence tensor %d NULL or misaligned", who, p);
    return DIT_OK;
}

}  // namespace
}  // namespace ditsp

using namespace ditsp;

extern "C" dit_status dit_ulysses_seq_to_head(const dit_sp_layout* L, int nplanes, const void* const* src,
                                              const void* const* src2, int split, dit_dtype src_dt,
                                              void* const* dst, const dit_dtype* dst_dt, const float* cos_tab,
                                              const float* sin_tab, unsigned rope_planes, int* d_range_flag,
                                              void* stream) {
    NvtxRange nvtx_range("dit_ulysses_seq_to_head");
    const char* who = "dit_ulysses_seq_to_head";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (nplanes < 1 || nplanes > 3) return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3", who);
    if (!dtype_ok(src_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad source dtype", who);
    if (!dst_dt) return fail(DIT_ERR_INVALID_ARG, "%s: dst_dt NULL", who);
    for (int p = 0; p < nplanes; ++p)
        if (!dtype_ok(dst_dt[p])) return fail(DIT_ERR_INVALID_ARG, "%s: bad destination dtype", who);
    if (split < 0 || split > L->S) return fail(DIT_ERR_INVALID_ARG, "%s: split out of [0, S]", who);
    if (rope_planes >> nplanes) return fail(DIT_ERR_INVALID_ARG, "%s: rope_planes names a missing plane", who);
    if (L->S == 0) return DIT_OK;
    if (rope_planes && (!cos_tab || !sin_tab || !aligned16(cos_tab) || !aligned16(sin_tab)))
        return fail(DIT_ERR_INVALID_ARG, "%s: rotary tables NULL or misaligned", who);
    if (!src || !dst) return fail(DIT_ERR_INVALID_ARG, "%s: src/dst NULL", who);
    if (split > 0 && split < L->S && !src2) return fail(DIT_ERR_INVALID_ARG, "%s: src2 NULL", who);
    DirectArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    for (int p = 0; p < nplanes; ++p) {
        if ((s = seq_pair_ok(src[p], src2 ? src2[p] : nullptr, split, L->S, who, p)) != DIT_OK) return s;
        if (!dst[p] || !aligned16(dst[p]))
            return fail(DIT_ERR_INVALID_ARG, "%s: dst[%d] NULL or misaligned", who, p);
        a.seq[p] = const_cast<char*>(static_cast<const char*>(src[p]));
        a.seq2[p] = src2 ? const_cast<char*>(static_cast<const char*>(src2[p])) : nullptr;
        a.head[p] = static_cast<char*>(dst[p]);
        a.src_dt[p] = src_dt;
        a.dst_dt[p] = dst_dt[p];
    }
    // a split at 0 or S leaves one tensor holding every row
    a.split = (split > 0 && split < L->S) ? split : 0;
    a.range_flag = d_range_flag;
    a.cos_tab = cos_tab;
    a.sin_tab = sin_tab;
    a.rope_planes = rope_planes;
    a.nrows = (long long)nplanes * L->B * L->S_pad;
    a.cpr = (int)(((long long)L->Hp * L->D) >> 3);
    a.creal = (int)(((long long)L->H * L->D) >> 3);
    const cudaStream_t st = (cudaStream_t)stream;
    return rope_planes ? launch_direct<true, true>(a, st, who) : launch_direct<true, false>(a, st, who);
}

extern "C" dit_status dit_ulysses_head_to_seq(const dit_sp_layout* L, const void* src, dit_dtype src_dt, void* dst,
                                              void* dst2, int split, dit_dtype dst_dt, void* stream) {
    NvtxRange nvtx_range("dit_ulysses_head_to_seq");
    const char* who = "dit_ulysses_head_to_seq";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!dtype_ok(src_dt) || !dtype_ok(dst_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (split < 0 || split > L->S) return fail(DIT_ERR_INVALID_ARG, "%s: split out of [0, S]", who);
    if (L->S == 0) return DIT_OK;
    if (!src || !aligned16(src)) return fail(DIT_ERR_INVALID_ARG, "%s: src NULL or misaligned", who);
    if ((s = seq_pair_ok(dst, dst2, split, L->S, who, 0)) != DIT_OK) return s;
    DirectArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = 1;
    a.head[0] = const_cast<char*>(static_cast<const char*>(src));
    a.seq[0] = static_cast<char*>(dst);
    a.seq2[0] = static_cast<char*>(dst2);
    a.split = (split > 0 && split < L->S) ? split : 0;
    a.src_dt[0] = src_dt;
    a.dst_dt[0] = dst_dt;
    a.nrows = (long long)L->B * L->S;
    a.cpr = (int)(((long long)L->H * L->D) >> 3);
    a.creal = a.cpr;
    return launch_direct<false, false>(a, (cudaStream_t)stream, who);
}
