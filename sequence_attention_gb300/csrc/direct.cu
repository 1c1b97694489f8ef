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
// Work division: the destination is a sequence of rows of cpr 8-element
// chunks, one row per warp; a row's source and destination addresses are the
// same for every lane (no per-chunk index arithmetic), and lanes take its
// chunks 32 apart.  Per batch of kDirItems chunks a lane issues every 16-byte
// load first, then converts and stores.  A rotated row's angle rows are
// staged in shared memory once per warp, so each chunk reads its cosines and
// sines from there.  The 16-bit-source and rotated forms are held to three
// blocks per SM (80 registers; 8 to 32 bytes of spill): ncu showed the
// two-block form with a fifth of the warps active and long-scoreboard stalls.
#include <string.h>

#include "convert.cuh"
#include "sp_index.cuh"

namespace ditsp {
namespace {

constexpr int kDirThreads = 256;
constexpr int kDirItems = 8;     // chunks per lane in flight
constexpr int kDirMaxRopeD = 384;   // largest head dim of the rotary path

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
    long long share;             // destination rows per warp
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

// Where destination row `row` reads from and writes to.  src is NULL for a
// sequence-padding row (seq -> head), which is written as zeros.
struct RowIO {
    const char* src;
    char* dst;
    int p, t;
};

template <bool S2H, int SB, int DB>
__device__ __forceinline__ RowIO row_io(const DirectArgs& A, long long row) {
    const dit_sp_layout& L = A.L;
    RowIO io;
    if (S2H) {
        const long long per_plane = (long long)L.B * L.S_pad;
        io.p = (int)(row / per_plane);
        const long long rem = row - io.p * per_plane;
        const int b = (int)(rem / L.S_pad);
        io.t = (int)(rem - (long long)b * L.S_pad);
        io.dst = A.head[io.p] + head_row_elems(L, b, io.t) * DB;
        io.src = io.t < L.S ? seq_row(A, A.seq, A.seq2, io.p, b, io.t, SB) : nullptr;
    } else {
        const int b = (int)(row / L.S);
        io.p = 0;
        io.t = (int)(row - (long long)b * L.S);
        io.src = A.head[0] + head_row_elems(L, b, io.t) * SB;
        io.dst = seq_row(A, A.seq, A.seq2, 0, b, io.t, DB);
    }
    return io;
}

// OCC4: a 64-register build (4 blocks per SM) of the 16-bit head -> seq
// pass, for grids between one wave of 3 and one wave of 4 blocks per SM.
template <bool S2H, int SB, int DB, bool ROPE, bool OCC4 = false>
__global__ void __launch_bounds__(kDirThreads, OCC4 ? 4 : ((ROPE || SB == 2) ? 3 : 1))
    direct_kernel(const __grid_constant__ DirectArgs A) {
    // rotary path: the token's cosine row then sine row (D/2 floats each),
    // staged per warp while the row's first data loads are in flight
    __shared__ float4 tab_sm[ROPE ? kDirThreads / 32 : 1][ROPE ? kDirMaxRopeD / 4 : 1];
    const dit_sp_layout& L = A.L;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long warp = (long long)blockIdx.x * (kDirThreads / 32) + wib;
    const long long row0 = warp * A.share;
    const long long row1 = min(A.nrows, row0 + A.share);
    pdl_wait();
    const bool want_check = S2H && A.range_flag != nullptr;
    bool overflow = false;
    constexpr int NI = kDirItems;
    const int q4 = L.D >> 3;                 // float4s per table row
    for (long long row = row0; row < row1; ++row) {
        // the row's place on both sides (the same for every lane of the warp)
        const RowIO io = row_io<S2H, SB, DB>(A, row);
        const int rp = io.p;
        const bool rreal = io.src != nullptr;
        const dit_dtype sdt = A.src_dt[rp], ddt = A.dst_dt[rp];
        const bool rot = ROPE && rreal && ((A.rope_planes >> rp) & 1u);
        const int lim = rreal ? A.creal : 0;     // chunks read from the source; the rest are zero
        if (ROPE && rot) {
            const float4* ct = reinterpret_cast<const float4*>(A.cos_tab + (long long)io.t * (L.D >> 1));
            const float4* sn = reinterpret_cast<const float4*>(A.sin_tab + (long long)io.t * (L.D >> 1));
            for (int j = lane; j < 2 * q4; j += 32) cp_async16(&tab_sm[wib][j], j < q4 ? ct + j : sn + (j - q4));
            cp_async_commit();
        }
        // every lane runs the same batches (the table staging has a warp barrier)
        for (int c0 = 0; c0 < A.cpr; c0 += 32 * NI) {
            uint4 raw[NI][SB / 2];
#pragma unroll
            for (int k = 0; k < NI; ++k) {
                const int c = c0 + lane + 32 * k;
#pragma unroll
                for (int h = 0; h < SB / 2; ++h) raw[k][h] = make_uint4(0, 0, 0, 0);
                if (c < lim) {
                    const uint4* src = reinterpret_cast<const uint4*>(io.src + (long long)c * 8 * SB);
#pragma unroll
                    for (int h = 0; h < SB / 2; ++h) raw[k][h] = src[h];
                }
            }
            if (ROPE && rot && c0 == 0) {
                cp_async_wait_all();
                __syncwarp();
            }
#pragma unroll
            for (int k = 0; k < NI; ++k) {
                const int c = c0 + lane + 32 * k;
                if (c >= A.cpr) break;
                uint4 o[DB / 2];
                if (ROPE && rot && c < lim) {
                    const int i4 = (((c * 8) % L.D) >> 3);
                    rope8<SB, DB>(raw[k], sdt, ddt, tab_sm[wib][i4], tab_sm[wib][q4 + i4], want_check && ddt != DIT_F32,
                                  o, overflow);
                } else {
                    convert8<SB, DB>(raw[k], sdt, ddt, want_check && narrowing(sdt, ddt), o, overflow);
                }
                uint4* d = reinterpret_cast<uint4*>(io.dst + (long long)c * 8 * DB);
#pragma unroll
                for (int h = 0; h < DB / 2; ++h) d[h] = o[h];
            }
        }
        if (ROPE && rot) __syncwarp();      // the next row's staging overwrites the tables
    }
    if (overflow) *A.range_flag = (int)DIT_ERR_RANGE;
    pdl_trigger();
}

template <bool S2H, int SB, int DB, bool ROPE>
dit_status launch_direct_sized(DirectArgs& a, cudaStream_t st, const char* who) {
    // one destination row per warp, as many blocks as that takes: the block
    // scheduler streams them through memory in order (measured against one
    // wave of resident warps with equal shares of rows and against a staged
    // form with bulk copies into shared memory: both slower, 5.3-5.9 TB/s
    // against 6.0 at the FLUX-like and 7.1 TB/s at the Wan-like size)
    a.share = 1;
    const long long blocks = (a.nrows + kDirThreads / 32 - 1) / (kDirThreads / 32);
    if (blocks >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: too many rows", who);
    cudaError_t e;
    // A 16-bit head -> seq grid just over one wave of 3 blocks per SM runs
    // in one wave of the 4-blocks-per-SM build (FLUX-like output, 576
    // blocks: 10.57 against 10.86 us back to back, same bits); over many
    // waves the 3-block build is faster (Wan-like: 223.4 against 226.2 us).
    if constexpr (!S2H && SB == 2 && !ROPE) {
        const long long nsm = num_sms();
        if (blocks > 3 * nsm && blocks <= 4 * nsm)
            e = launch_pdl(direct_kernel<S2H, SB, DB, ROPE, true>, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a);
        else
            e = launch_pdl(direct_kernel<S2H, SB, DB, ROPE>, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a);
    } else {
        e = launch_pdl(direct_kernel<S2H, SB, DB, ROPE>, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a);
    }
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

// ---- the three-call path's seq -> head unpack, one head-layout row per warp
// Head-layout row (plane p, ring block r, batch b, row t - ring_off[r]) holds
// Hp heads that arrive as U runs of the receive wire (order B): run v is
// head_len[v] heads of D elements at slot slots_B(p, b, t, v).  With U <= 32
// lane v keeps run v's start, less head_off[v]*D, so chunk c (8 elements,
// c*8 into the row) reads wire element base(v(c)) + c*8, with v(c) the group
// of head c*8/D (a multiply-shift division when every group has Hl heads);
// with more ranks each chunk computes its run's start itself.  Chunks of real
// heads of real rows are rotated when the plane is; the rest are copied
// (zeros on the wire).  Same arithmetic as the run-walking unpack, so the
// same bits.
struct WireArgs {
    dit_sp_layout L;
    int np;
    const char* wire;
    char* head[3];
    dit_dtype src_dt, dst_dt[3];
    int* range_flag;
    const float* cos_tab;
    const float* sin_tab;
    unsigned rope_planes;
    long long nrows;             // np * B * S_pad
    int cpr;                     // chunks per head-layout row (Hp * D / 8)
    int creal;                   // chunks of real heads (H * D / 8)
    FastDiv head_of;             // chunk -> head (D / 8 chunks a head)
    FastDiv group_of;            // head -> group when every group has Hl heads
    int even;
};

template <int SB, int DB, bool ROPE>
__global__ void __launch_bounds__(kDirThreads, SB == 2 ? 3 : 1) wire_unpack_kernel(const __grid_constant__ WireArgs A) {
    __shared__ float4 tab_sm[ROPE ? kDirThreads / 32 : 1][ROPE ? kDirMaxRopeD / 4 : 1];
    const dit_sp_layout& L = A.L;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long row = (long long)blockIdx.x * (kDirThreads / 32) + wib;
    pdl_wait();
    if (row >= A.nrows) {      // no block barrier below: a warp may leave
        pdl_trigger();
        return;
    }
    const long long per_plane = (long long)L.B * L.S_pad;
    const int p = (int)(row / per_plane);
    const long long rem = row - p * per_plane;
    const int b = (int)(rem / L.S_pad), t = (int)(rem - (long long)b * L.S_pad);
    Run x;
    const int rid = rank_of_row(L, t);
    x.r = rid / L.U;
    x.u = rid - x.r * L.U;
    x.p = p;
    x.b = b;
    x.i = t - L.rank_off[rid];
    char* dst = A.head[p] + ((((long long)x.r * L.B + b) * L.S_cap + (t - L.ring_off[x.r])) * L.Hp) * L.D * DB;
    long long base = 0;        // lane v: run v's first wire element, less head_off[v] * D
    if (lane < L.U && lane < 32) {
        x.v = lane;
        base = slots_B(L, A.np, x) * L.D - (long long)L.head_off[lane] * L.D;
    }
    const dit_dtype sdt = A.src_dt, ddt = A.dst_dt[p];
    const bool rot = ROPE && t < L.S && ((A.rope_planes >> p) & 1u);
    const int rlim = rot ? A.creal : 0;          // chunks rotated
    const bool want_check = A.range_flag != nullptr && narrowing(sdt, ddt);
    const bool want_check_rot = A.range_flag != nullptr && ddt != DIT_F32;
    bool overflow = false;
    const int q4 = L.D >> 3;
    if (ROPE && rot) {
        const float4* ct = reinterpret_cast<const float4*>(A.cos_tab + (long long)t * (L.D >> 1));
        const float4* sn = reinterpret_cast<const float4*>(A.sin_tab + (long long)t * (L.D >> 1));
        for (int j = lane; j < 2 * q4; j += 32) cp_async16(&tab_sm[wib][j], j < q4 ? ct + j : sn + (j - q4));
        cp_async_commit();
    }
    constexpr int NI = kDirItems;
    for (int c0 = 0; c0 < A.cpr; c0 += 32 * NI) {        // every lane runs the same batches
        uint4 raw[NI][SB / 2];
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int c = c0 + lane + 32 * k;
            const int h = (int)fdiv((uint32_t)min(c, A.cpr - 1), A.head_of);
            int v;
            if (A.even) {
                v = (int)fdiv((uint32_t)h, A.group_of);
            } else {
                int lo = 0, hi = L.U - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (L.head_off[mid] <= h) lo = mid; else hi = mid - 1;
                }
                v = lo;
            }
            long long src;
            if (L.U <= 32) {                                 // warp-uniform
                src = __shfl_sync(0xffffffffu, base, v);
            } else {
                Run y = x;
                y.v = v;
                src = slots_B(L, A.np, y) * L.D - (long long)L.head_off[v] * L.D;
            }
#pragma unroll
            for (int e = 0; e < SB / 2; ++e) raw[k][e] = make_uint4(0, 0, 0, 0);
            if (c < A.cpr) {
                const uint4* g = reinterpret_cast<const uint4*>(A.wire + (src + (long long)c * 8) * SB);
#pragma unroll
                for (int e = 0; e < SB / 2; ++e) raw[k][e] = g[e];
            }
        }
        if (ROPE && rot && c0 == 0) {
            cp_async_wait_all();
            __syncwarp();
        }
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int c = c0 + lane + 32 * k;
            if (c >= A.cpr) break;
            uint4 o[DB / 2];
            if (ROPE && c < rlim) {
                const int i4 = c - (int)fdiv((uint32_t)c, A.head_of) * q4;
                rope8<SB, DB>(raw[k], sdt, ddt, tab_sm[wib][i4], tab_sm[wib][q4 + i4], want_check_rot, o, overflow);
            } else {
                convert8<SB, DB>(raw[k], sdt, ddt, want_check, o, overflow);
            }
            uint4* d = reinterpret_cast<uint4*>(dst + (long long)c * 8 * DB);
#pragma unroll
            for (int e = 0; e < DB / 2; ++e) d[e] = o[e];
        }
    }
    if (ROPE && rot) __syncwarp();
    if (overflow) *A.range_flag = (int)DIT_ERR_RANGE;
    pdl_trigger();
}

template <int SB, int DB, bool ROPE>
dit_status launch_wire(const WireArgs& a, cudaStream_t st, const char* who) {
    const long long blocks = (a.nrows + kDirThreads / 32 - 1) / (kDirThreads / 32);
    if (blocks >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: too many rows", who);
    cudaError_t e = launch_pdl(wire_unpack_kernel<SB, DB, ROPE>, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

template <bool ROPE>
dit_status launch_wire_typed(const WireArgs& a, cudaStream_t st, const char* who) {
    const int sb = dtype_bytes(a.src_dt), db = dtype_bytes(a.dst_dt[0]);
    if (sb == 2 && db == 2) return launch_wire<2, 2, ROPE>(a, st, who);
    if (sb == 4 && db == 4) return launch_wire<4, 4, ROPE>(a, st, who);
    if (sb == 4 && db == 2) return launch_wire<4, 2, ROPE>(a, st, who);
    return launch_wire<2, 4, ROPE>(a, st, who);
}

// ---- the three-call path's seq -> head exchange, one sequence row per warp
// Row (plane p, batch b, padded-sequence row t) of the send wire (order A)
// holds U runs, run v at slots_A(p, b, t, v); the exchange copies each to
// slots_B(p, b, t, v) of the receive wire (order B).  Lane v keeps both
// starts less head_off[v]*D, so chunk c of the row (8 elements) moves from
// src(v(c)) + c*8 to dst(v(c)) + c*8, v(c) found as in wire_unpack_kernel.
// A raw copy (e4m3 records travel as (D + 16) / 2 16-bit words).
struct CopyArgs {
    dit_sp_layout L;             // D = elements (or 16-bit words) a head slot
    int np;
    const char* src;
    char* dst;
    long long nrows;             // np * B * S_pad
    int cpr;                     // chunks per row (Hp * D / 8)
    FastDiv head_of;
    FastDiv group_of;
    int even;
};

template <int EB>
__global__ void __launch_bounds__(kDirThreads, EB == 2 ? 3 : 1) wire_a2a_kernel(const __grid_constant__ CopyArgs A) {
    const dit_sp_layout& L = A.L;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * (kDirThreads / 32) + (threadIdx.x >> 5);
    pdl_wait();
    if (row >= A.nrows) {
        pdl_trigger();
        return;
    }
    const long long per_plane = (long long)L.B * L.S_pad;
    const int p = (int)(row / per_plane);
    const long long rem = row - p * per_plane;
    const int b = (int)(rem / L.S_pad), t = (int)(rem - (long long)b * L.S_pad);
    Run x;
    const int rid = rank_of_row(L, t);
    x.r = rid / L.U;
    x.u = rid - x.r * L.U;
    x.p = p;
    x.b = b;
    x.i = t - L.rank_off[rid];
    long long sa = 0, sb = 0;  // lane v: run v's starts on both wires, less head_off[v] * D
    if (lane < L.U && lane < 32) {
        x.v = lane;
        const long long back = (long long)L.head_off[lane] * L.D;
        sa = slots_A(L, A.np, x) * L.D - back;
        sb = slots_B(L, A.np, x) * L.D - back;
    }
    constexpr int NI = kDirItems;
    for (int c0 = 0; c0 < A.cpr; c0 += 32 * NI) {
        uint4 raw[NI][EB / 2];
        long long to[NI];
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int c = c0 + lane + 32 * k;
            const int h = (int)fdiv((uint32_t)min(c, A.cpr - 1), A.head_of);
            int v;
            if (A.even) {
                v = (int)fdiv((uint32_t)h, A.group_of);
            } else {
                int lo = 0, hi = L.U - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (L.head_off[mid] <= h) lo = mid; else hi = mid - 1;
                }
                v = lo;
            }
            long long from;
            if (L.U <= 32) {                                 // warp-uniform
                from = __shfl_sync(0xffffffffu, sa, v);
                to[k] = __shfl_sync(0xffffffffu, sb, v);
            } else {
                Run y = x;
                y.v = v;
                const long long back = (long long)L.head_off[v] * L.D;
                from = slots_A(L, A.np, y) * L.D - back;
                to[k] = slots_B(L, A.np, y) * L.D - back;
            }
            from += (long long)c * 8;
            to[k] += (long long)c * 8;
#pragma unroll
            for (int e = 0; e < EB / 2; ++e) raw[k][e] = make_uint4(0, 0, 0, 0);
            if (c < A.cpr) {
                const uint4* g = reinterpret_cast<const uint4*>(A.src + from * EB);
#pragma unroll
                for (int e = 0; e < EB / 2; ++e) raw[k][e] = g[e];
            }
        }
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int c = c0 + lane + 32 * k;
            if (c >= A.cpr) break;
            uint4* d = reinterpret_cast<uint4*>(A.dst + to[k] * EB);
#pragma unroll
            for (int e = 0; e < EB / 2; ++e) d[e] = raw[k][e];
        }
    }
    pdl_trigger();
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

// The three-call seq -> head exchange: see wire_a2a_kernel.  Lw is the
// layout with D = the head slot's width in units of eb bytes (2 or 4).
dit_status wire_a2a_s2h(const dit_sp_layout* Lw, int nplanes, const void* send, void* recv, int eb,
                        cudaStream_t st, const char* who) {
    if (Lw->U > 64) return fail(DIT_ERR_UNSUPPORTED, "%s: more than 64 Ulysses ranks", who);
    CopyArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *Lw;
    a.np = nplanes;
    a.src = static_cast<const char*>(send);
    a.dst = static_cast<char*>(recv);
    a.nrows = (long long)nplanes * Lw->B * Lw->S_pad;
    a.cpr = (int)(((long long)Lw->Hp * Lw->D) >> 3);
    a.head_of = make_fastdiv((uint32_t)(Lw->D >> 3));
    a.even = 1;
    for (int v = 0; v < Lw->U; ++v) a.even &= Lw->head_len[v] == Lw->Hl && Lw->head_off[v] == v * Lw->Hl;
    a.group_of = make_fastdiv((uint32_t)(Lw->Hl > 0 ? Lw->Hl : 1));
    if (a.nrows == 0) return DIT_OK;
    const long long blocks = (a.nrows + kDirThreads / 32 - 1) / (kDirThreads / 32);
    if (blocks >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: too many rows", who);
    cudaError_t e = eb == 4 ? launch_pdl(wire_a2a_kernel<4>, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a)
                            : launch_pdl(wire_a2a_kernel<2>, dim3((unsigned)blocks), dim3(kDirThreads), 0, st, a);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

// The three-call seq -> head unpack (16/32-bit wire), optional RoPE: see
// wire_unpack_kernel.  Arguments are validated by the callers.
dit_status wire_unpack_s2h(const dit_sp_layout* L, int nplanes, const void* recv, dit_dtype wire_dt,
                           void* const* dst, const dit_dtype* dst_dt, const float* cos_tab, const float* sin_tab,
                           unsigned rope_planes, int* range_flag, cudaStream_t st, const char* who) {
    const int db = dtype_bytes(dst_dt[0]);
    for (int p = 1; p < nplanes; ++p)
        if (dtype_bytes(dst_dt[p]) != db)
            return fail(DIT_ERR_UNSUPPORTED, "%s: planes of one call need destination types of one size", who);
    if (rope_planes && L->D > kDirMaxRopeD)
        return fail(DIT_ERR_UNSUPPORTED, "%s: the rotary path supports D <= %d", who, kDirMaxRopeD);
    if (L->U > 64) return fail(DIT_ERR_UNSUPPORTED, "%s: more than 64 Ulysses ranks", who);
    WireArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    a.wire = static_cast<const char*>(recv);
    for (int p = 0; p < nplanes; ++p) {
        a.head[p] = static_cast<char*>(dst[p]);
        a.dst_dt[p] = dst_dt[p];
    }
    a.src_dt = wire_dt;
    a.range_flag = range_flag;
    a.cos_tab = cos_tab;
    a.sin_tab = sin_tab;
    a.rope_planes = rope_planes;
    a.nrows = (long long)nplanes * L->B * L->S_pad;
    a.cpr = (int)(((long long)L->Hp * L->D) >> 3);
    a.creal = (int)(((long long)L->H * L->D) >> 3);
    a.head_of = make_fastdiv((uint32_t)(L->D >> 3));
    a.even = 1;
    for (int v = 0; v < L->U; ++v) a.even &= L->head_len[v] == L->Hl && L->head_off[v] == v * L->Hl;
    a.group_of = make_fastdiv((uint32_t)(L->Hl > 0 ? L->Hl : 1));
    if (a.nrows == 0) return DIT_OK;
    return rope_planes ? launch_wire_typed<true>(a, st, who) : launch_wire_typed<false>(a, st, who);
}

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
    if (rope_planes && L->D > kDirMaxRopeD)
        return fail(DIT_ERR_UNSUPPORTED, "%s: the rotary path supports D <= %d", who, kDirMaxRopeD);
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
