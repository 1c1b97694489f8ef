// Index arithmetic of the Ulysses exchange, shared by the 16/32-bit
// permutation kernels and the FP8-wire kernels.
//
// A "run" is the head group of one rank for one (plane, batch, row): the
// head_len[v] head slots of Ulysses rank v, head_len[v]*D contiguous
// elements on every side of the exchange.  Two wire orders exist; in units
// of head slots (Hp = all slots, Hv = head_len[v], ov = head_off[v]):
//   A (sequence side): rank (r,u)'s buffer = for v: [planes][B][L_u] runs
//      np*B*Hp*off_u + np*B*L_u*ov + ((p*B+b)*L_u + i)*Hv
//   B (head side):     rank (r,v)'s buffer = for u: [planes][B][L_u] runs
//      np*B*Hp*off_r + np*B*S_r*ov + np*B*(off_u-off_r)*Hv + ((p*B+b)*L_u + i)*Hv
// Runs are numbered in either order without regard to their sizes (A: rank,
// v, plane, batch, row; B: ring block, v, u, plane, batch, row).
// Seq-to-head: pack writes A, the exchange copies A->B, unpack reads B.
// Head-to-seq: pack writes B, the exchange copies B->A, unpack reads A.
// Rows are those of the padded sequence (S_pad); rows at or past S are
// sequence padding.
#pragma once

#include "common.cuh"

namespace ditsp {
namespace {

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

// Run index -> (r, u, v, p, b, i).  All run counts fit in 32 bits (checked
// on the host), so the divisions here are 32-bit.
__device__ __forceinline__ Run decode_A(const dit_sp_layout& L, int np, int a) {
    const int per_row = np * L.B * L.U;
    const int rid = rank_of_row(L, a / per_row);
    Run x;
    x.r = rid / L.U; x.u = rid - x.r * L.U;
    const int Lu = L.rank_len[rid];
    const int local = a - per_row * L.rank_off[rid];
    const int blk = np * L.B * Lu;
    x.v = local / blk;
    const int rem = local - x.v * blk;
    const int pb = rem / Lu;
    x.i = rem - pb * Lu;
    x.p = pb / L.B; x.b = pb - x.p * L.B;
    return x;
}

__device__ __forceinline__ Run decode_B(const dit_sp_layout& L, int np, int bi) {
    const int per_row = np * L.B * L.U;
    Run x;
    x.r = ring_of_row(L, bi / per_row);
    const int offr = L.ring_off[x.r];
    const int grp = np * L.B * L.ring_len[x.r];
    const int local = bi - per_row * offr;
    x.v = local / grp;
    int rem = local - x.v * grp;
    const int rid = rank_of_row(L, offr + rem / (np * L.B));
    x.u = rid - x.r * L.U;
    const int Lu = L.rank_len[rid];
    rem -= np * L.B * (L.rank_off[rid] - offr);
    const int pb = rem / Lu;
    x.i = rem - pb * Lu;
    x.p = pb / L.B; x.b = pb - x.p * L.B;
    return x;
}

// Head-layout order (destination order of the seq->head unpack): runs of
// plane p enumerated as (r, b, row of ring block r, v), so consecutive runs
// fill one head-layout row.
__device__ __forceinline__ Run decode_H(const dit_sp_layout& L, int np, int h) {
    const int per_plane = L.B * L.S_pad * L.U;
    Run x;
    x.p = h / per_plane;
    const int rem = h - x.p * per_plane;
    x.r = ring_of_row(L, rem / (L.B * L.U));
    const int offr = L.ring_off[x.r], Sr = L.ring_len[x.r];
    const int local = rem - L.B * L.U * offr;
    x.b = local / (Sr * L.U);
    const int rem2 = local - x.b * Sr * L.U;
    const int row = rem2 / L.U;
    x.v = rem2 - row * L.U;
    const int rid = rank_of_row(L, offr + row);
    x.u = rid - x.r * L.U;
    x.i = offr + row - L.rank_off[rid];
    return x;
}

// Sequence order (destination order of the head->seq unpack, one plane):
// runs enumerated as (b, token, v) over the S real tokens, so consecutive
// runs fill one token row.
__device__ __forceinline__ Run decode_S(const dit_sp_layout& L, int s) {
    Run x;
    x.p = 0;
    const int bt = s / L.U;
    x.v = s - bt * L.U;
    x.b = bt / L.S;
    const int t = bt - x.b * L.S;
    const int rid = rank_of_row(L, t);
    x.r = rid / L.U;
    x.u = rid - x.r * L.U;
    x.i = t - L.rank_off[rid];
    return x;
}

// Offset of a run in wire order A / B, in head slots.
__device__ __forceinline__ long long slots_A(const dit_sp_layout& L, int np, const Run& x) {
    const int rid = x.r * L.U + x.u;
    const long long Lu = L.rank_len[rid];
    return (long long)np * L.B * L.Hp * L.rank_off[rid] + np * L.B * Lu * L.head_off[x.v] +
           (((long long)x.p * L.B + x.b) * Lu + x.i) * L.head_len[x.v];
}

__device__ __forceinline__ long long slots_B(const dit_sp_layout& L, int np, const Run& x) {
    const int rid = x.r * L.U + x.u;
    const int offr = L.ring_off[x.r];
    const long long Hv = L.head_len[x.v];
    return (long long)np * L.B * L.Hp * offr + (long long)np * L.B * L.ring_len[x.r] * L.head_off[x.v] +
           (long long)np * L.B * (L.rank_off[rid] - offr) * Hv +
           (((long long)x.p * L.B + x.b) * L.rank_len[rid] + x.i) * Hv;
}

// global (padded-sequence) row of a run
__device__ __forceinline__ int run_row(const dit_sp_layout& L, const Run& x) {
    return L.rank_off[x.r * L.U + x.u] + x.i;
}

// head slots of the run's group that hold real heads (global head < H)
__device__ __forceinline__ int real_heads(const dit_sp_layout& L, int v) {
    return min(max(L.H - L.head_off[v], 0), L.head_len[v]);
}

// element offset of the run's first head in a seq-layout plane [B][S][H][D]
// (only meaningful when the group has a real head and the row is real).
// With paired streams,
// rows at or past `split` are in the second tensor, [B][S - split][H][D];
// `second` says which.
__device__ __forceinline__ long long seq_offset(const dit_sp_layout& L, const Run& x, int split, bool& second) {
    int row = L.rank_off[x.r * L.U + x.u] + x.i;
    int rows = L.S;
    second = split > 0 && row >= split;
    if (split > 0) {
        rows = second ? L.S - split : split;
        if (second) row -= split;
    }
    return (((long long)x.b * rows + row) * L.H + L.head_off[x.v]) * L.D;
}

// element offset in a head-layout plane [R][B][S_cap][Hp][D]
__device__ __forceinline__ long long head_offset(const dit_sp_layout& L, const Run& x) {
    const int row = L.rank_off[x.r * L.U + x.u] - L.ring_off[x.r] + x.i;
    return ((((long long)x.r * L.B + x.b) * L.S_cap + row) * L.Hp + L.head_off[x.v]) * L.D;
}

}  // namespace

// Host-side check of a caller-supplied layout (defined in ulysses.cu).
dit_status check_layout(const dit_sp_layout* L, const char* who);

// The e4m3 wire (fp8_wire.cu).  fp8_pack quantizes nplanes source planes
// (S2H; src2/split: paired streams, split 0 = one stream) or one head-layout
// tensor (H2S) into records; fp8_unpack decodes records into head-layout
// planes (S2H, optional RoPE on rope_planes) or the sequence layout (H2S,
// paired streams as for the pack).  Arguments are validated by the callers
// except the head dim, which must be a power of two in [16, 256].
dit_status fp8_pack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes, const void* const* src,
                    const void* const* src2, int split, dit_dtype src_dt, void* send, cudaStream_t st,
                    const char* who);
// The three-call seq -> head exchange as a copy of each sequence row's U runs
// from send order A to receive order B (direct.cu); Lw->D is the head slot's
// width in units of eb (2 or 4) bytes.
dit_status wire_a2a_s2h(const dit_sp_layout* Lw, int nplanes, const void* send, void* recv, int eb,
                        cudaStream_t st, const char* who);
// The three-call seq -> head unpack of a 16/32-bit wire into head-layout
// planes, one head-layout row per warp, optional RoPE on rope_planes
// (direct.cu).  Arguments are validated by the callers except the plane
// types' sizes and the rotary head dim.
dit_status wire_unpack_s2h(const dit_sp_layout* L, int nplanes, const void* recv, dit_dtype wire_dt,
                           void* const* dst, const dit_dtype* dst_dt, const float* cos_tab, const float* sin_tab,
                           unsigned rope_planes, int* range_flag, cudaStream_t st, const char* who);
dit_status fp8_unpack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes, const void* recv, void* const* dst,
                      void* const* dst2, int split, const dit_dtype* dst_dt, const float* cos_tab,
                      const float* sin_tab, unsigned rope_planes, int* range_flag, cudaStream_t st,
                      const char* who);

}  // namespace ditsp
