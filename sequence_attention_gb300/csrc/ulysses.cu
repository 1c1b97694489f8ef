// The Ulysses all-to-all as permutation kernels over virtual ranks that live
// in one GPU's memory (edge-dit.cpp "Parallel execution": packed QKV send
// path, receive preparation, head-to-sequence path; SGLang Diffusion
// "Parallelism Overview", The Ulysses transport: an all-to-all is a
// permutation, so a copy in one memory is bit-identical to any transport).
//
// Every buffer in the exchange is a sequence of "runs": the head_len[v]*D
// contiguous elements of one rank's head group v for one (plane, batch,
// row).  A run is contiguous on both sides of every step, so each kernel
// moves whole runs with 16-byte vectors: a warp takes a few runs, lanes over
// 8-element chunks.  The wire orders A (sequence side) and B (head side) and
// the offsets of a run in them are written out in sp_index.cuh.
// Seq-to-head: pack writes A, the exchange copies A->B, unpack reads B.
// Head-to-seq: pack writes B, the exchange copies B->A, unpack reads A.
// Each kernel walks the runs in its destination's order (A, B, head-layout
// or sequence order), so its writes are sequential and its reads gather.
// Rows of the padded sequence at or past S (lcm(SP, 64) padding) travel as
// zeros and are never read from or written to the sequence-layout tensors.
//
// Two additions of the receive preparation and of the FLUX double-stream
// blocks (edge-dit.cpp "Parallel execution"):
//  - paired streams: the sequence side of a call may live in two tensors,
//    text rows [0, split) and image rows [split, S) of the joint sequence,
//    so that the pack assembles the joint sequence and the head-to-seq
//    unpack splits it again without a concatenation or a slice copy;
//  - rotary embedding: the seq-to-head unpack may rotate chosen planes
//    (Q, K) while it writes the head layout, each interleaved pair (2i, 2i+1)
//    of a token at joint position t by the angle whose cosine and sine are
//    cos[t][i], sin[t][i]:  (x0, x1) -> (x0 c - x1 s, x0 s + x1 c), in fp32.
#include <string.h>

#include "convert.cuh"
#include "sp_index.cuh"

namespace ditsp {
namespace {

// The seq -> head unpack is the row-per-warp wire_unpack_s2h (direct.cu).
enum Mode { PACK_S2H = 0, UNPACK_H2S, PACK_H2S, A2A_S2H, A2A_H2S };

struct RunArgs {
    dit_sp_layout L;
    int np;
    const void* src[3];
    void* dst[3];
    dit_dtype src_dt[3];
    dit_dtype dst_dt[3];
    int* range_flag;
    long long nruns;
    // checked exchange: copy a run only once its sender's counter reached epoch
    const unsigned* arrival;
    unsigned epoch;
    long long timeout_ns;
    int* status;
    // paired streams (split > 0): sequence-side rows t >= split live in
    // src2/dst2 at row t - split; split == 0 means a single stream
    const void* src2[3];
    void* dst2[3];
    int split;
};

__device__ __forceinline__ unsigned long long gtimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Publish `epoch` on the arrival counter of every rank whose bit is set.
__global__ void signal_kernel(unsigned* arrival, int nranks, unsigned long long mask, unsigned epoch) {
    pdl_wait();
    const int i = threadIdx.x;
    if (i < nranks && ((mask >> i) & 1ull)) {
        __threadfence();
        arrival[i] = epoch;
    }
    pdl_trigger();
}

// Where one run comes from and goes to (chunk = 8 elements).
struct RunIO {
    const char* src;
    char* dst;
    int src_lim;      // chunks of the source holding data; later chunks read as zero
    int dst_lim;      // chunks of the destination written; later chunks skipped
    int sdt, ddt;     // dit_dtype of source and destination
    int sender;       // virtual rank that sent this run (exchange kernels)
};

template <int MODE>
__device__ __forceinline__ RunIO run_io(const RunArgs& A, int ri) {
    const dit_sp_layout& L = A.L;
    // Every kernel enumerates runs in the order of its destination, so that
    // consecutive runs write consecutive memory.
    Run x;
    if (MODE == PACK_S2H || MODE == A2A_H2S) x = decode_A(L, A.np, ri);
    else if (MODE == UNPACK_H2S) x = decode_S(L, ri);
    else x = decode_B(L, A.np, ri);
    const int p = x.p;
    const long long D = L.D;
    // head slots of this run, and those holding real heads; a row at or past
    // S is sequence padding and holds none
    const bool pad_row = run_row(L, x) >= L.S;
    const int nreal = pad_row ? 0 : real_heads(L, x.v);
    const int full = (L.head_len[x.v] * L.D) >> 3, real = (nreal * L.D) >> 3;
    RunIO io;
    io.src_lim = io.dst_lim = full;
    long long so = 0, doff = 0;
    dit_dtype sdt, ddt;
    bool second = false;
    if (MODE == PACK_S2H) {
        sdt = A.src_dt[p]; ddt = A.dst_dt[0];
        so = nreal > 0 ? seq_offset(L, x, A.split, second) : 0; doff = slots_A(L, A.np, x) * D;
        io.src = (const char*)(second ? A.src2[p] : A.src[p]); io.dst = (char*)A.dst[0];
        io.src_lim = real;
    } else if (MODE == UNPACK_H2S) {
        sdt = A.src_dt[0]; ddt = A.dst_dt[0];
        so = slots_A(L, A.np, x) * D; doff = nreal > 0 ? seq_offset(L, x, A.split, second) : 0;
        io.src = (const char*)A.src[0]; io.dst = (char*)(second ? A.dst2[0] : A.dst[0]);
        io.dst_lim = real;
    } else if (MODE == PACK_H2S) {
        sdt = A.src_dt[0]; ddt = A.dst_dt[0];
        so = head_offset(L, x); doff = slots_B(L, A.np, x) * D;
        io.src = (const char*)A.src[0]; io.dst = (char*)A.dst[0];
        io.src_lim = real;
    } else if (MODE == A2A_S2H) {
        sdt = ddt = A.src_dt[0];
        so = slots_A(L, A.np, x) * D; doff = slots_B(L, A.np, x) * D;
        io.src = (const char*)A.src[0]; io.dst = (char*)A.dst[0];
    } else {  // A2A_H2S
        sdt = ddt = A.src_dt[0];
        so = slots_B(L, A.np, x) * D; doff = slots_A(L, A.np, x) * D;
        io.src = (const char*)A.src[0]; io.dst = (char*)A.dst[0];
    }
    io.src += so * dtype_bytes(sdt);
    io.dst += doff * dtype_bytes(ddt);
    io.sdt = sdt;
    io.ddt = ddt;
    // seq->head: rank (r,u) sends to (r,v); head->seq: rank (r,v) sends to (r,u)
    io.sender = x.r * L.U + (MODE == A2A_H2S || MODE == PACK_H2S || MODE == UNPACK_H2S ? x.v : x.u);
    (void)ri;
    return io;
}


constexpr int kThreads = 256;
constexpr int kItems = 8;       // 8-element items per lane in flight

// Each block takes 8 * rpw consecutive runs (rpw = runs per warp, 4, or 2
// for small exchanges): threads decode
// one run each into shared memory, then each warp streams its rpw runs,
// lanes over their 8-element chunks.  Per group of kItems items a lane
// issues every load first, converts in registers, then stores.
template <int MODE, int SB, int DB>
__global__ void __launch_bounds__(kThreads, 1) run_kernel(const __grid_constant__ RunArgs A, int rpw) {
    __shared__ RunIO ios[kThreads];
    const int rpb = rpw * (kThreads / 32);
    const long long r0 = (long long)blockIdx.x * rpb;
    const int nrun = (int)min((long long)rpb, A.nruns - r0);
    if ((int)threadIdx.x < nrun) ios[threadIdx.x] = run_io<MODE>(A, (int)(r0 + threadIdx.x));
    __syncthreads();
    pdl_wait();          // the decode above used only the layout; data from here on
    if (A.arrival != nullptr && (int)threadIdx.x < nrun) {
        // Bounded wait for the sender's arrival counter (a transport whose
        // peer never publishes must fail, not hang).  Once any wait of the
        // call has run out, every other run is abandoned at once.
        RunIO& io = ios[threadIdx.x];
        const volatile unsigned* cnt = A.arrival + io.sender;
        volatile int* st = A.status;
        bool arrived = (int)(*cnt - A.epoch) >= 0;
        if (!arrived) {
            const unsigned long long t0 = gtimer_ns();
            while (!arrived && *st != (int)DIT_ERR_TIMEOUT) {
                __nanosleep(256);
                arrived = (int)(*cnt - A.epoch) >= 0;
                if (!arrived && gtimer_ns() - t0 > (unsigned long long)A.timeout_ns) {
                    atomicExch(A.status, (int)DIT_ERR_TIMEOUT);
                    break;
                }
            }
        }
        if (!arrived) io.src_lim = io.dst_lim = 0;
        // the counter was read relaxed: order this thread's observation of
        // the sender's release before the block's loads of the send buffer
        else __threadfence();
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g0 = warp * rpw;
    const int gn = min(rpw, nrun - g0);
    if (gn <= 0) {
        pdl_trigger();
        return;
    }
    const int nch = (A.L.Hl * A.L.D) >> 3;
    const int items = gn > 0 ? gn * nch : 0;
    constexpr int NI = kItems;
    int g = lane / nch, c = lane - (lane / nch) * nch;   // item k0 = lane
    uint4 raw[NI][SB / 2];
    // item t of a batch: run g0 + (it[t] >> 16), chunk it[t] & 0xffff
    // (fewer than 2^16 chunks per run, checked on the host)
    int it[NI];
    auto load_batch = [&](int k0) {
#pragma unroll
        for (int t = 0; t < NI; ++t) {
            it[t] = (g << 16) | c;
            c += 32;
            while (c >= nch) { c -= nch; ++g; }
        }
#pragma unroll
        for (int t = 0; t < NI; ++t) {
#pragma unroll
            for (int h = 0; h < SB / 2; ++h) raw[t][h] = make_uint4(0, 0, 0, 0);
            if (k0 + 32 * t < items) {
                const int ci = it[t] & 0xffff;
                const RunIO& io = ios[g0 + (it[t] >> 16)];
                if (ci < io.src_lim) {
                    const uint4* q = reinterpret_cast<const uint4*>(io.src + (long long)ci * 8 * SB);
#pragma unroll
                    for (int h = 0; h < SB / 2; ++h) raw[t][h] = q[h];
                }
            }
        }
    };
    auto store_batch = [&](int k0) {
#pragma unroll
        for (int t = 0; t < NI; ++t) {
            if (k0 + 32 * t < items) {
                const int gi = it[t] >> 16, ci = it[t] & 0xffff;
                const RunIO& io = ios[g0 + gi];
                if (ci < io.dst_lim) {
                    const dit_dtype sdt = (dit_dtype)io.sdt, ddt = (dit_dtype)io.ddt;
                    uint4 o[DB / 2];
                    bool unused = false;     // no narrowing to check off the seq -> head unpack
                    convert8<SB, DB>(raw[t], sdt, ddt, false, o, unused);
                    uint4* q = reinterpret_cast<uint4*>(io.dst + (long long)ci * 8 * DB);
#pragma unroll
                    for (int h = 0; h < DB / 2; ++h) q[h] = o[h];
                }
            }
        }
    };
    for (int k0 = lane; k0 < items; k0 += 32 * NI) {
        load_batch(k0);
        store_batch(k0);
    }
    pdl_trigger();
}

template <int MODE, int SB, int DB>
dit_status launch_sized(const RunArgs& a, cudaStream_t st, const char* who) {
    // Up to 8 runs per warp (64 per block): measured on the FLUX-like step
    // against 1, 2, 3, 4, 6, 12, 16, 24 and 32, 8 gives the shortest layout
    // steps (layout-in 5.8, layout-out 5.7 TB/s) and the fastest Wan-size
    // unpacks; smaller blocks pay their run decoding too often, larger ones
    // leave the last wave uneven.  Small exchanges take fewer runs per warp so
    // that the grid still has about two blocks per SM.
    long long fit = a.nruns / (16LL * num_sms());
    const int rpw = fit < 1 ? 1 : (fit > 8 ? 8 : (int)fit);
    const long long blocks = (a.nruns + 8LL * rpw - 1) / (8LL * rpw);
    cudaError_t e = launch_pdl(run_kernel<MODE, SB, DB>, dim3((unsigned)blocks), dim3(kThreads), 0, st, a, rpw);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

// Element sizes are template parameters so that 16-bit paths hold 16-byte
// items; every plane of one call must use source (and destination) types
// of one size.
template <int MODE>
dit_status launch_runs(const RunArgs& a, cudaStream_t st, const char* who) {
    if (a.nruns == 0) return DIT_OK;
    if (a.nruns >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: more than 2^31 runs", who);
    if ((long long)a.L.Hl * a.L.D / 8 >= (1LL << 16))
        return fail(DIT_ERR_UNSUPPORTED, "%s: a head group holds 2^19 or more elements", who);
    const int sb = dtype_bytes(a.src_dt[0]);
    const int db = dtype_bytes(a.dst_dt[0]);
    for (int p = 1; p < 3; ++p) {
        if (a.src[p] && dtype_bytes(a.src_dt[p]) != sb)
            return fail(DIT_ERR_UNSUPPORTED, "%s: planes of one call need source types of one size", who);
        if (a.dst[p] && dtype_bytes(a.dst_dt[p]) != db)
            return fail(DIT_ERR_UNSUPPORTED, "%s: planes of one call need destination types of one size", who);
    }
    if (sb == 2 && db == 2) return launch_sized<MODE, 2, 2>(a, st, who);
    if (sb == 4 && db == 4) return launch_sized<MODE, 4, 4>(a, st, who);
    if (sb == 4 && db == 2) return launch_sized<MODE, 4, 2>(a, st, who);
    return launch_sized<MODE, 2, 4>(a, st, who);
}

}  // namespace

// The e4m3 wire's exchange: a record of D + 16 bytes is (D + 16) / 2 16-bit
// words, so the exchange is the 16-bit permutation of runs of that width.
static dit_status check_e4m3_dim(int D, const char* who) {
    if (D < 16 || D > 256 || (D & (D - 1)))
        return fail(DIT_ERR_UNSUPPORTED, "%s: the e4m3 wire needs D in {16, 32, 64, 128, 256}", who);
    return DIT_OK;
}

// A layout with S = 0 has no rows on either side of the exchange: the call
// moves nothing, launches nothing and does not look at its buffer pointers
// (an allocator may give NULL for zero bytes).  The e4m3 wire's head-dim
// rule is still checked, so the answer does not depend on S.
static dit_status empty_exchange(const dit_sp_layout* L, dit_dtype wire_dt, const char* who) {
    return wire_dt == DIT_E4M3 ? check_e4m3_dim(L->D, who) : DIT_OK;
}

dit_status record_words(RunArgs* a, const char* who) {
    const int D = a->L.D;
    const dit_status s = check_e4m3_dim(D, who);
    if (s != DIT_OK) return s;
    a->L.D = (D + 16) / 2;
    a->src_dt[0] = a->dst_dt[0] = DIT_BF16;
    return DIT_OK;
}

// Host-side check of a caller-supplied layout: every field must be what
// dit_sp_layout_init would have produced for its (B, S, H, D, U, R).
dit_status check_layout(const dit_sp_layout* L, const char* who) {
    if (!L) return fail(DIT_ERR_INVALID_ARG, "%s: layout is NULL", who);
    dit_sp_layout ref;
    if (dit_sp_layout_init_ex(L->B, L->S, L->H, L->D, L->U, L->R, L->flags, &ref) != DIT_OK)
        return fail(DIT_ERR_INVALID_ARG, "%s: layout sizes invalid", who);
    bool ok = ref.Hp == L->Hp && ref.Hl == L->Hl && ref.S_cap == L->S_cap && ref.S_pad == L->S_pad;
    for (int v = 0; ok && v < L->U; ++v)
        ok = ref.head_len[v] == L->head_len[v] && ref.head_off[v] == L->head_off[v];
    for (int r = 0; ok && r < L->R; ++r)
        ok = ref.ring_len[r] == L->ring_len[r] && ref.ring_off[r] == L->ring_off[r] &&
             ref.ring_real[r] == L->ring_real[r];
    for (int i = 0; ok && i < L->R * L->U; ++i)
        ok = ref.rank_len[i] == L->rank_len[i] && ref.rank_off[i] == L->rank_off[i];
    if (!ok) return fail(DIT_ERR_INVALID_ARG, "%s: layout tables are inconsistent", who);
    if (L->D % 8 != 0)
        return fail(DIT_ERR_UNSUPPORTED, "%s: head dim %d is not a multiple of 8", who, L->D);
    return DIT_OK;
}

}  // namespace ditsp

using namespace ditsp;

extern "C" dit_status dit_ulysses_pack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                       const void* const* src, dit_dtype src_dt, void* send,
                                       dit_dtype wire_dt, void* stream) {
    NvtxRange nvtx_range("dit_ulysses_pack");
    const char* who = "dit_ulysses_pack";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!dtype_ok(src_dt) || !wire_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3 || (dir == DIT_HEAD_TO_SEQ && nplanes != 1))
        return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3 (1 for head-to-seq)", who);
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
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
    a.nruns = (long long)nplanes * L->B * L->U * L->S_pad;
    cudaStream_t st = (cudaStream_t)stream;
    if (wire_dt == DIT_E4M3) return fp8_pack(L, dir, nplanes, src, nullptr, 0, src_dt, send, st, who);
    return dir == DIT_SEQ_TO_HEAD ? launch_runs<PACK_S2H>(a, st, who) : launch_runs<PACK_H2S>(a, st, who);
}

extern "C" dit_status dit_a2a_sim(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                  const void* send, void* recv, dit_dtype wire_dt, void* stream) {
    NvtxRange nvtx_range("dit_a2a_sim");
    const char* who = "dit_a2a_sim";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!wire_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3) return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3", who);
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
    if (!send || !recv || !aligned16(send) || !aligned16(recv) || send == recv)
        return fail(DIT_ERR_INVALID_ARG, "%s: send/recv NULL, misaligned or identical", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    a.src[0] = send; a.src_dt[0] = wire_dt;
    a.dst[0] = recv; a.dst_dt[0] = wire_dt;
    a.nruns = (long long)nplanes * L->B * L->U * L->S_pad;
    if (wire_dt == DIT_E4M3 && (s = record_words(&a, who)) != DIT_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (dir == DIT_SEQ_TO_HEAD) return wire_a2a_s2h(&a.L, nplanes, send, recv, dtype_bytes(a.src_dt[0]), st, who);
    return launch_runs<A2A_H2S>(a, st, who);
}

extern "C" dit_status dit_ulysses_unpack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                         const void* recv, dit_dtype wire_dt, void* const* dst,
                                         const dit_dtype* dst_dt, int* d_range_flag, void* stream) {
    NvtxRange nvtx_range("dit_ulysses_unpack");
    const char* who = "dit_ulysses_unpack";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!wire_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad wire dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3 || (dir == DIT_HEAD_TO_SEQ && nplanes != 1))
        return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3 (1 for head-to-seq)", who);
    if (!dst_dt) return fail(DIT_ERR_INVALID_ARG, "%s: dst_dt NULL", who);
    for (int p = 0; p < nplanes; ++p)
        if (!dtype_ok(dst_dt[p])) return fail(DIT_ERR_INVALID_ARG, "%s: bad dst dtype", who);
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
    if (!recv || !aligned16(recv) || !dst)
        return fail(DIT_ERR_INVALID_ARG, "%s: recv/dst NULL or misaligned", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    a.src[0] = recv; a.src_dt[0] = wire_dt;
    for (int p = 0; p < nplanes; ++p) {
        if (!dst[p] || !aligned16(dst[p])) return fail(DIT_ERR_INVALID_ARG, "%s: dst[%d] NULL or misaligned", who, p);
        a.dst[p] = dst[p];
        a.dst_dt[p] = dst_dt[p];
    }
    a.range_flag = d_range_flag;
    a.nruns = (long long)nplanes * L->B * L->U * (dir == DIT_SEQ_TO_HEAD ? L->S_pad : L->S);
    cudaStream_t st = (cudaStream_t)stream;
    if (wire_dt == DIT_E4M3)
        return fp8_unpack(L, dir, nplanes, recv, dst, nullptr, 0, dst_dt, nullptr, nullptr, 0, d_range_flag, st, who);
    if (dir == DIT_SEQ_TO_HEAD)
        return wire_unpack_s2h(L, nplanes, recv, wire_dt, dst, dst_dt, nullptr, nullptr, 0, d_range_flag, st, who);
    return launch_runs<UNPACK_H2S>(a, st, who);
}

extern "C" dit_status dit_sp_signal(const dit_sp_layout* L, unsigned* d_arrival, const unsigned char* rank_mask,
                                    unsigned epoch, void* stream) {
    NvtxRange nvtx_range("dit_sp_signal");
    const char* who = "dit_sp_signal";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!d_arrival || (reinterpret_cast<uintptr_t>(d_arrival) & 3))
        return fail(DIT_ERR_INVALID_ARG, "%s: arrival counters NULL or misaligned", who);
    const int n = L->U * L->R;
    unsigned long long mask = 0;
    for (int i = 0; i < n; ++i)
        if (!rank_mask || rank_mask[i]) mask |= 1ull << i;
    cudaError_t e = launch_pdl(signal_kernel, dim3(1), dim3(64), 0, (cudaStream_t)stream, d_arrival, n, mask, epoch);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

extern "C" dit_status dit_a2a_sim_checked(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes, const void* send,
                                          void* recv, dit_dtype wire_dt, const unsigned* d_arrival, unsigned epoch,
                                          int64_t timeout_ns, int* d_status, void* stream) {
    NvtxRange nvtx_range("dit_a2a_sim_checked");
    const char* who = "dit_a2a_sim_checked";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!wire_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (dir != DIT_SEQ_TO_HEAD && dir != DIT_HEAD_TO_SEQ) return fail(DIT_ERR_INVALID_ARG, "%s: bad direction", who);
    if (nplanes < 1 || nplanes > 3) return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3", who);
    if (!d_arrival || (reinterpret_cast<uintptr_t>(d_arrival) & 3))
        return fail(DIT_ERR_INVALID_ARG, "%s: arrival counters NULL or misaligned", who);
    if (timeout_ns <= 0 || timeout_ns > 10000000000LL)
        return fail(DIT_ERR_INVALID_ARG, "%s: timeout must be in (0, 10 s]", who);
    // nothing is read, so nothing waits for the senders
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
    if (!send || !recv || !aligned16(send) || !aligned16(recv) || send == recv)
        return fail(DIT_ERR_INVALID_ARG, "%s: send/recv NULL, misaligned or identical", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    a.src[0] = send; a.src_dt[0] = wire_dt;
    a.dst[0] = recv; a.dst_dt[0] = wire_dt;
    a.nruns = (long long)nplanes * L->B * L->U * L->S_pad;
    a.arrival = d_arrival;
    a.epoch = epoch;
    a.timeout_ns = timeout_ns;
    a.status = d_status ? d_status : default_status_word();
    if (!a.status) return fail(DIT_ERR_CUDA, "%s: no device status word", who);
    if (wire_dt == DIT_E4M3 && (s = record_words(&a, who)) != DIT_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    return dir == DIT_SEQ_TO_HEAD ? launch_runs<A2A_S2H>(a, st, who) : launch_runs<A2A_H2S>(a, st, who);
}

extern "C" dit_status dit_ulysses_pack_joint(const dit_sp_layout* L, int nplanes, const void* const* txt,
                                             const void* const* img, int S_txt, dit_dtype src_dt, void* send,
                                             dit_dtype wire_dt, void* stream) {
    NvtxRange nvtx_range("dit_ulysses_pack_joint");
    const char* who = "dit_ulysses_pack_joint";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!dtype_ok(src_dt) || !wire_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (nplanes < 1 || nplanes > 3) return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3", who);
    if (S_txt < 0 || S_txt > L->S) return fail(DIT_ERR_INVALID_ARG, "%s: S_txt out of [0, S]", who);
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
    if (!send || !aligned16(send)) return fail(DIT_ERR_INVALID_ARG, "%s: send NULL or misaligned", who);
    const bool has_txt = S_txt > 0, has_img = S_txt < L->S;
    if ((has_txt && !txt) || (has_img && !img)) return fail(DIT_ERR_INVALID_ARG, "%s: stream array NULL", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = nplanes;
    for (int p = 0; p < nplanes; ++p) {
        if (has_txt && (!txt[p] || !aligned16(txt[p])))
            return fail(DIT_ERR_INVALID_ARG, "%s: txt[%d] NULL or misaligned", who, p);
        if (has_img && (!img[p] || !aligned16(img[p])))
            return fail(DIT_ERR_INVALID_ARG, "%s: img[%d] NULL or misaligned", who, p);
        // one stream only: it is the whole sequence
        a.src[p] = has_txt ? txt[p] : img[p];
        a.src2[p] = has_txt && has_img ? img[p] : nullptr;
        a.src_dt[p] = src_dt;
    }
    a.split = has_txt && has_img ? S_txt : 0;
    a.dst[0] = send;
    a.dst_dt[0] = wire_dt;
    a.nruns = (long long)nplanes * L->B * L->U * L->S_pad;
    if (wire_dt == DIT_E4M3)
        return fp8_pack(L, DIT_SEQ_TO_HEAD, nplanes, a.src, a.src2, a.split, src_dt, send, (cudaStream_t)stream, who);
    return launch_runs<PACK_S2H>(a, (cudaStream_t)stream, who);
}

extern "C" dit_status dit_ulysses_unpack_joint(const dit_sp_layout* L, const void* recv, dit_dtype wire_dt,
                                               void* out_txt, void* out_img, int S_txt, dit_dtype out_dt,
                                               void* stream) {
    NvtxRange nvtx_range("dit_ulysses_unpack_joint");
    const char* who = "dit_ulysses_unpack_joint";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!wire_ok(wire_dt) || !dtype_ok(out_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (S_txt < 0 || S_txt > L->S) return fail(DIT_ERR_INVALID_ARG, "%s: S_txt out of [0, S]", who);
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
    if (!recv || !aligned16(recv)) return fail(DIT_ERR_INVALID_ARG, "%s: recv NULL or misaligned", who);
    const bool has_txt = S_txt > 0, has_img = S_txt < L->S;
    if ((has_txt && (!out_txt || !aligned16(out_txt))) || (has_img && (!out_img || !aligned16(out_img))))
        return fail(DIT_ERR_INVALID_ARG, "%s: output stream NULL or misaligned", who);
    RunArgs a;
    memset(&a, 0, sizeof(a));
    a.L = *L;
    a.np = 1;
    a.src[0] = recv; a.src_dt[0] = wire_dt;
    a.dst[0] = has_txt ? out_txt : out_img;
    a.dst2[0] = has_txt && has_img ? out_img : nullptr;
    a.dst_dt[0] = out_dt;
    a.split = has_txt && has_img ? S_txt : 0;
    a.nruns = (long long)L->B * L->U * L->S;
    if (wire_dt == DIT_E4M3)
        return fp8_unpack(L, DIT_HEAD_TO_SEQ, 1, recv, a.dst, a.dst2, a.split, a.dst_dt, nullptr, nullptr, 0, nullptr,
                          (cudaStream_t)stream, who);
    return launch_runs<UNPACK_H2S>(a, (cudaStream_t)stream, who);
}

extern "C" dit_status dit_ulysses_unpack_rope(const dit_sp_layout* L, int nplanes, const void* recv,
                                              dit_dtype wire_dt, void* const* dst, const dit_dtype* dst_dt,
                                              const float* cos_tab, const float* sin_tab, unsigned rope_planes,
                                              int* d_range_flag, void* stream) {
    NvtxRange nvtx_range("dit_ulysses_unpack_rope");
    const char* who = "dit_ulysses_unpack_rope";
    dit_status s = check_layout(L, who);
    if (s != DIT_OK) return s;
    if (!wire_ok(wire_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad wire dtype", who);
    if (nplanes < 1 || nplanes > 3) return fail(DIT_ERR_INVALID_ARG, "%s: nplanes must be 1..3", who);
    if (rope_planes >> nplanes) return fail(DIT_ERR_INVALID_ARG, "%s: rope_planes names a missing plane", who);
    if (!dst_dt) return fail(DIT_ERR_INVALID_ARG, "%s: dst_dt NULL", who);
    for (int p = 0; p < nplanes; ++p)
        if (!dtype_ok(dst_dt[p])) return fail(DIT_ERR_INVALID_ARG, "%s: bad dst dtype", who);
    if (L->S == 0) return empty_exchange(L, wire_dt, who);
    if (rope_planes && (!cos_tab || !sin_tab || !aligned16(cos_tab) || !aligned16(sin_tab)))
        return fail(DIT_ERR_INVALID_ARG, "%s: rotary tables NULL or misaligned", who);
    if (!recv || !aligned16(recv) || !dst)
        return fail(DIT_ERR_INVALID_ARG, "%s: recv/dst NULL or misaligned", who);
    for (int p = 0; p < nplanes; ++p)
        if (!dst[p] || !aligned16(dst[p])) return fail(DIT_ERR_INVALID_ARG, "%s: dst[%d] NULL or misaligned", who, p);
    cudaStream_t st = (cudaStream_t)stream;
    if (wire_dt == DIT_E4M3)
        return fp8_unpack(L, DIT_SEQ_TO_HEAD, nplanes, recv, dst, nullptr, 0, dst_dt, cos_tab, sin_tab, rope_planes,
                          d_range_flag, st, who);
    return wire_unpack_s2h(L, nplanes, recv, wire_dt, dst, dst_dt, cos_tab, sin_tab, rope_planes, d_range_flag, st,
                           who);
}
