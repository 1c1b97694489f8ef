// Attention partial on the Blackwell tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, per (query block r, key/value block j, batch b, head h), the
// attention of Q_r against the valid keys of (K_j, V_j) with the row
// log-sum-exp (SGLang Diffusion "Parallelism Overview", Constraints: the
// ring merge needs each call's softmax LSE; edge-dit.cpp "Parallel
// execution": exact full-sequence attention per head).
//
// CTA = 256 query rows as two 128-row tiles of one (query block r, batch
// b, head h); the CTA walks every key block j of r in turn (with diag, block
// r only) and writes partial (r, j) at the end of block j.  Warp roles:
//   warps 0-3  softmax for Q tile 0 (TMEM lanes 0-127, one row per thread)
//   warps 4-7  softmax for Q tile 1
//   warp  8    TMA producer of Q (once) and K tiles (2-stage ring); halfway
//              through, the L2 prefetch of the next wave's first tiles
//   warp  9    MMA issuer (one thread): S = Q K^T and O += P V
//   warp  10   TMA producer of V tiles (2-stage ring); K and V loads wait on
//              their own ring's releases, so neither holds up the other
//   warp  11   idle (completes the third warpgroup)
// Registers: launched at 168 per thread; the producer/MMA warpgroup gives
// back down to 104 and the two softmax warpgroups take 200 each
// (2*200 + 104 = 3*168), enough to hold a whole 128-column score row.
// TMEM (512 columns x 128 lanes, fp32): S0 [0,128) S1 [128,256)
// O0 [256,256+D) O1 [256+D,256+2D).  P (16-bit) overwrites the first half
// of its tile's S columns and feeds the P V MMA straight from TMEM.
//
// Per key tile the MMA thread issues, for the two Q tiles in turn:
// P V for tile t of key tile n, then Q K^T for tile t of key tile n+1, so
// the tensor core computes one tile's products while the other tile's
// softmax runs.  Softmax keeps the row max in the log2 domain and only
// rescales the O accumulator when a row's max grows by more than 2^8
// (values of P stay <= 256, exact in f16/bf16 and fp32); the final 1/l
// normalisation uses the same reference max, so the result is exact up to
// rounding.  Keys at or past the block's valid length are masked to -inf;
// TMA zero-fills rows past each block's extent, so padding bytes in the
// buffers are never read.
// The epilogue writes O / l through a per-warp shared-memory slot and TMA
// stores, each warp its 32 rows; the output map has the block's own extents,
// so no row past the block is written.
//
// Every mbarrier wait is bounded (a few seconds of %globaltimer); on expiry
// the CTA records DIT_ERR_TIMEOUT in the status word, stops issuing work,
// waits (bounded) for the copies and MMAs it already issued, frees TMEM and
// exits.
#include <math.h>
#include <string.h>

#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"

namespace ditsp {
namespace {

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 128;          // keys per tile (MMA N of Q K^T, K of P V)
constexpr int NQT = 2;           // query tiles per CTA
constexpr int NSK = 2;           // K pipeline stages
// V pipeline stages: 2 (the third tile's worth of shared memory holds the
// per-warp output staging slots)
constexpr int kNSV = 2;
constexpr int kSlot = 32 * 128;  // one warp's staging slot: 32 rows x 128 bytes
constexpr int NTHREADS = 384;
constexpr int CHUNK = BM * 128;  // bytes of one 64-column (128-byte) swizzle chunk
constexpr unsigned long long kWaitNs = 4000000000ull;

// Barriers.  Position g of the walk (key tile g over every block) consumes
// the pair (K tile g+1, V tile g) -- what P V(g) and Q K^T(g+1) read -- and
// the pair lands on one full barrier B_F + g % 2 and is released by one
// commit on B_E + g % 2; K tile 0 lands with Q on B_Q.
enum { B_Q = 0, B_F = 1, B_E = 3, B_SF = 5, B_PF = 7, B_OD = 9, B_END = 11, NBAR = 12 };

struct TcParams {
    CUtensorMap qmap[DIT_MAX_R];
    CUtensorMap kmap[DIT_MAX_R];
    CUtensorMap vmap[DIT_MAX_R];
    CUtensorMap omap[DIT_MAX_R];    // output of query block r: (d, h, row, b, key block)
    int q_len[DIT_MAX_R];
    int kv_len[DIT_MAX_R];
    int q_row0[DIT_MAX_R];          // first output row of query block r (packed sequences)
    int o_row0[DIT_MAX_R];          // further rows into o of query block r's output
    int B, n_q, n_kv;
    int diag;                       // query block r attends key block r only
    int fold;                       // one output per query block: the key blocks folded by the online softmax
    int nsm;                        // SMs of the device (CTAs in flight: one per SM)
    float c;                      // scale * log2(e)
    uint32_t idesc_qk, idesc_pv;
    dit_view o;
    dit_dtype o_dt;
    dit_lse_view lse;
    int* status;
};

// shared memory: Q tiles | K stages | V stages | staging slots | barriers
template <int D>
__host__ __device__ constexpr int bars_offset() {
    return (NQT + NSK + kNSV) * BM * D * 2 + 8 * kSlot;
}
template <int D>
__host__ __device__ constexpr int smem_bytes() {
    return bars_offset<D>() + NBAR * 8 + 16 + 1024;
}

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The CTA's abort flag (a shared-memory word, by its 32-bit shared address)
// and the caller's status word.
struct Ctl {
    uint32_t abort;
    int* status;
};
__device__ __forceinline__ int ld_flag(uint32_t a) {
    int v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_flag(uint32_t a, int v) {
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Wait for the phase of `parity` to complete.  Returns false if the CTA has
// aborted or this wait ran out of time (then the CTA is marked aborted).
__device__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl& ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (ld_flag(ctl.abort)) return false;
            if (gtimer() - t0 > kWaitNs) {
                st_flag(ctl.abort, 1);
                atomicExch(ctl.status, (int)DIT_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: used to drain work already
// issued before the CTA frees its resources.
__device__ void drain_phase(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = gtimer();
    while (!mbar_try_wait(bar, parity))
        if (gtimer() - t0 > kWaitNs) return;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Shared -> global tile store of one 128-byte-wide box (rows past the map's
// extent are not written), and the bulk-group completion wait.
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3,
                                             int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading/stride byte offsets in 16-byte units, version 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// TMEM <-> register moves of 32-bit columns of this thread's lane.  Each load
// carries its wait in the same asm block, so no use of the registers can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&x)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&x)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31]), "=r"(x[32]), "=r"(x[33]), "=r"(x[34]), "=r"(x[35]), "=r"(x[36]), "=r"(x[37]), "=r"(x[38]), "=r"(x[39]), "=r"(x[40]), "=r"(x[41]), "=r"(x[42]), "=r"(x[43]), "=r"(x[44]), "=r"(x[45]), "=r"(x[46]), "=r"(x[47]), "=r"(x[48]), "=r"(x[49]), "=r"(x[50]), "=r"(x[51]), "=r"(x[52]), "=r"(x[53]), "=r"(x[54]), "=r"(x[55]), "=r"(x[56]), "=r"(x[57]), "=r"(x[58]), "=r"(x[59]), "=r"(x[60]), "=r"(x[61]), "=r"(x[62]), "=r"(x[63])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&x)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31]), "=r"(x[32]), "=r"(x[33]), "=r"(x[34]), "=r"(x[35]), "=r"(x[36]), "=r"(x[37]), "=r"(x[38]), "=r"(x[39]), "=r"(x[40]), "=r"(x[41]), "=r"(x[42]), "=r"(x[43]), "=r"(x[44]), "=r"(x[45]), "=r"(x[46]), "=r"(x[47]), "=r"(x[48]), "=r"(x[49]), "=r"(x[50]), "=r"(x[51]), "=r"(x[52]), "=r"(x[53]), "=r"(x[54]), "=r"(x[55]), "=r"(x[56]), "=r"(x[57]), "=r"(x[58]), "=r"(x[59]), "=r"(x[60]), "=r"(x[61]), "=r"(x[62]), "=r"(x[63]), "=r"(x[64]), "=r"(x[65]), "=r"(x[66]), "=r"(x[67]), "=r"(x[68]), "=r"(x[69]), "=r"(x[70]), "=r"(x[71]), "=r"(x[72]), "=r"(x[73]), "=r"(x[74]), "=r"(x[75]), "=r"(x[76]), "=r"(x[77]), "=r"(x[78]), "=r"(x[79]), "=r"(x[80]), "=r"(x[81]), "=r"(x[82]), "=r"(x[83]), "=r"(x[84]), "=r"(x[85]), "=r"(x[86]), "=r"(x[87]), "=r"(x[88]), "=r"(x[89]), "=r"(x[90]), "=r"(x[91]), "=r"(x[92]), "=r"(x[93]), "=r"(x[94]), "=r"(x[95]), "=r"(x[96]), "=r"(x[97]), "=r"(x[98]), "=r"(x[99]), "=r"(x[100]), "=r"(x[101]), "=r"(x[102]), "=r"(x[103]), "=r"(x[104]), "=r"(x[105]), "=r"(x[106]), "=r"(x[107]), "=r"(x[108]), "=r"(x[109]), "=r"(x[110]), "=r"(x[111]), "=r"(x[112]), "=r"(x[113]), "=r"(x[114]), "=r"(x[115]), "=r"(x[116]), "=r"(x[117]), "=r"(x[118]), "=r"(x[119]), "=r"(x[120]), "=r"(x[121]), "=r"(x[122]), "=r"(x[123]), "=r"(x[124]), "=r"(x[125]), "=r"(x[126]), "=r"(x[127])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&x)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr), "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]), "r"(x[16]), "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]), "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31]) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
    if (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// The CTA's query block r, key block j, batch b, head h and first query row.
// %ctaid is read with volatile moves, so the epilogue recomputes these rather
// than keeping them live (in registers the softmax needs) through the
// key-tile loop.
// The CTA covers every key block of (r, b), starting at j (0, or r with
// DIAG, where query block r attends key block r only).
struct Cta {
    int r, j, b, h, row_base;
};
template <bool DIAG>
__device__ __forceinline__ Cta cta_coords(const TcParams& p) {
    uint32_t x, y, z;
    asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(x));
    asm volatile("mov.u32 %0, %%ctaid.y;" : "=r"(y));
    asm volatile("mov.u32 %0, %%ctaid.z;" : "=r"(z));
    Cta c;
    c.b = (int)z % p.B;
    c.r = (int)z / p.B;
    c.j = DIAG ? c.r : 0;
    c.h = (int)y;
    c.row_base = (int)x * (NQT * BM);
    return c;
}

// The partial (r, j) of an empty key block: O = 0 and lse = -inf for the
// CTA's rows, one row per thread of the two softmax warpgroups.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// The CTAs of a wave run in step: they all start, and fetch their Q and the
// first K and V tiles of new heads from DRAM, at once, while in the key loop
// K and V come from L2 and DRAM idles.  Halfway through its key loop a CTA
// therefore prefetches into L2 what the first Q K^T and P V of the CTA one
// SM count further in launch order read (usually one of the next wave):
// both Q tiles and the first K and V tiles.  A hint only; nothing waits on
// it.
template <int D, bool DIAG>
__device__ __forceinline__ void prefetch_next_cta(const TcParams& p) {
    const unsigned long long gx = gridDim.x, gy = gridDim.y, gz = gridDim.z;
    const unsigned long long L = blockIdx.x + gx * (blockIdx.y + gy * blockIdx.z) + (unsigned long long)p.nsm;
    if (L >= gx * gy * gz) return;
    const int x = (int)(L % gx), h = (int)((L / gx) % gy), z = (int)(L / (gx * gy));
    const int b = z % p.B, r = z / p.B;
    int j = r;                       // with DIAG, else the walk's first block with keys
    if (!DIAG) {
        for (j = 0; j < p.n_kv && p.kv_len[j] == 0; ++j) {
        }
        if (j == p.n_kv) return;
    }
    const int row_base = x * (NQT * BM);
    if (row_base >= p.q_len[r] || p.kv_len[j] == 0) return;
    for (int c = 0; c < D / 64; ++c) {
        for (int t = 0; t < NQT; ++t) tma_prefetch_4d(&p.qmap[r], c * 64, h, row_base + t * BM, b);
        tma_prefetch_4d(&p.kmap[j], c * 64, h, 0, b);
        tma_prefetch_4d(&p.vmap[j], c * 64, h, 0, b);
    }
}

template <int D>
__device__ __forceinline__ void write_empty_partial(const TcParams& p, int r, int j, int b, int h, int row_base) {
    if (threadIdx.x >= NQT * BM) return;
    const int row = row_base + (int)threadIdx.x;
    if (row >= p.q_len[r]) return;
    const int eb = dtype_bytes(p.o_dt);
    char* orow = static_cast<char*>(p.o.ptr) + (r * p.o.stride_q + j * p.o.stride_kv + b * p.o.stride_b +
                                                h * p.o.stride_h +
                                                ((long long)p.q_row0[r] + p.o_row0[r] + row) * p.o.stride_s) * eb;
    for (int d = 0; d < D; d += 8) store8_zero(orow + d * eb, p.o_dt);
    if (p.lse.ptr)
        p.lse.ptr[r * p.lse.stride_q + j * p.lse.stride_kv + b * p.lse.stride_b + h * p.lse.stride_h + p.q_row0[r] +
                  row] = -INFINITY;
}

// One key tile of the online softmax for the calling thread's query row
// (its TMEM lane): S (fp32, columns St) becomes P (16-bit, written over the
// first half of S); the reference max m (log2 domain) and the row sum l are
// updated, and O (columns Ot) is rescaled when the row max grows by more
// than 2^8, so P stays <= 256.  Keys at or past `valid` are masked to -inf;
// `first` marks the first tile of a key block.  Returns once P and any O
// rescale are in TMEM and ordered before the caller's "P written" arrive.
template <int D, bool P_BF16>
__device__ __forceinline__ void softmax_tile(uint32_t St, uint32_t Ot, int valid, bool first, float c, float& m_used,
                                             float& l) {
    uint32_t x[BN];
    tmem_ld128(St, x);                       // the whole score row, one round trip
    if (valid < BN) {                        // keys past the block: -inf
#pragma unroll
        for (int e = 0; e < BN; ++e)
            if (e >= valid) x[e] = 0xff800000u;
    }
    // row max: 8 independent chains of three-input max over columns 8 .. BN-9,
    // then the last 8 columns with a two-input max
    static_assert(BN % 16 == 0, "the max chains take 16 columns per step");
    float m8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(x[e]);
#pragma unroll
    for (int e = 8; e + 16 <= BN; e += 16)
#pragma unroll
        for (int q = 0; q < 8; ++q) m8[q] = max3(m8[q], __uint_as_float(x[e + q]), __uint_as_float(x[e + 8 + q]));
#pragma unroll
    for (int q = 0; q < 8; ++q) m8[q] = fmaxf(m8[q], __uint_as_float(x[BN - 8 + q]));
    const float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
    const float mxs = mx * c;
    float alpha = 1.f;
    bool rescale = false;
    if (first) {
        m_used = mxs;
    } else if (__any_sync(0xffffffffu, mxs > m_used + 8.f)) {
        // Raise the reference max; O is rescaled below, after P is written
        // (this tile's P V is not issued before the caller's arrive).
        const float mnew = fmaxf(m_used, mxs);
        alpha = ex2(m_used - mnew);
        m_used = mnew;
        rescale = true;
    }
    // P = 2^(s*c - m) (packed fp32 pairs), row sum in 4 packed chains, P
    // written over S in two halves
    const float2 c2 = make_float2(c, c), negm2 = make_float2(-m_used, -m_used);
    float2 l2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) l2[e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        // each half's TMEM store runs while the next half is computed
        uint32_t pk[BN / 4];
#pragma unroll
        for (int e = 0; e < BN / 4; ++e) {
            const int i0 = half * (BN / 2) + 2 * e;
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(x[i0]), __uint_as_float(x[i0 + 1])), c2, negm2);
            const float2 pp = make_float2(ex2(a.x), ex2(a.y));
            l2[e & 3] = __fadd2_rn(l2[e & 3], pp);
            pk[e] = pack_p<P_BF16>(pp.x, pp.y);
        }
        tmem_st32(St + half * (BN / 4), pk);
    }
    l = fmaf(l, alpha, ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y)) + ((l2[2].x + l2[2].y) + (l2[3].x + l2[3].y)));
    if (rescale) {
        // the previous P V of this tile completed before S became ready
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t y[32];
            tmem_ld32(Ot + cc * 32, y);
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = __float_as_uint(__uint_as_float(y[e]) * alpha);
            tmem_st32(Ot + cc * 32, y);
        }
    }
    tmem_wait_st();
    tc_fence_before();
}

// ---- the kernels ------------------------------------------------------------
// attn_tc_kernel: the CTA walks every key block j of its query rows in turn
// (with diag, block r only), keeping Q resident, and writes partial (r, j)
// at the end of block j; the K/V rings, the S/P barriers and the MMA stream
// run on without a break across the blocks, so the pipeline fills and
// drains once per CTA instead of once per block.  Warp roles: 0-7 softmax
// (two warpgroups, one query tile each), 8 the TMA producer, 9 the MMA
// issuer.  K and V have 2 stages each; the third tile's worth of shared
// memory holds one output staging slot per softmax warp, since the Q, K and
// V buffers stay in use until the last block.
template <int D, bool P_BF16, bool DIAG, bool FOLD>
__global__ void __launch_bounds__(NTHREADS, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
    static_assert(!(DIAG && FOLD), "folding walks every key block");
    constexpr int NCH = D / 64;          // 128-byte chunks per row
    constexpr int TILE = BM * D * 2;     // bytes of one Q, K or V tile
    constexpr int NSV = kNSV;
    static_assert(NSV == 2 && NSK == 2, "pairs (K g+1, V g) use stage g % 2 of both rings");
    constexpr int BARS = bars_offset<D>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + NQT * TILE;
    uint8_t* sV = sK + NSK * TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BARS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Cta cta = cta_coords<DIAG>(p);
    const int b = cta.b, r = cta.r, h = cta.h, row_base = cta.row_base;
    // key blocks j0 .. j0 + nj - 1 (j0 = cta.j: 0, or r with DIAG)
    const int nj = DIAG ? 1 : p.n_kv;
    if (row_base >= p.q_len[r]) return;
    bool any_keys = false;
    for (int jj = 0; jj < nj; ++jj) any_keys |= p.kv_len[cta.j + jj] > 0;
    if (!any_keys) {     // every key block empty: O = 0, lse = -inf
        pdl_wait();
        for (int jj = 0; jj < (FOLD ? 1 : nj); ++jj) write_empty_partial<D>(p, r, cta.j + jj, b, h, row_base);
        return;
    }

    const Ctl ctl{su32(const_cast<int*>(abort_flag)), p.status};
    auto bar = [&](int i) { return su32(bars + i); };

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_F + s), 1);
            mbar_init(bar(B_E + s), 1);
        }
        for (int t = 0; t < NQT; ++t) {
            mbar_init(bar(B_SF + t), 1);
            mbar_init(bar(B_PF + t), 128);
            mbar_init(bar(B_OD + t), 1);
        }
        mbar_init(bar(B_END), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();          // barriers and TMEM are set up; tensors from here on

    if (warp >= 8) {
        // the walking MMA issuer keeps more loop state: 104 registers here,
        // 200 for each softmax warpgroup (2*200 + 104 = 3*168)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
        if (warp == 8) {
        // ------------------------------------------------------------ producer
        // Key tiles are numbered across the key blocks (g); K tile g sits in
        // K stage g % 2, V tile g in V stage g % 2.  Pair g = (K g+1, V g)
        // waits until pair g-2's buffers are released (pair -1 is K tile 0,
        // released after the first Q K^T of both query tiles).
        if (lane == 0) {
            const int j0 = cta.j;
            int total = 0;                                  // key tiles over every block
            for (int jj = 0; jj < nj; ++jj) total += (p.kv_len[j0 + jj] + BN - 1) / BN;
            // cursor over the walk's key tiles: block jj, tile n (empty blocks skipped)
            struct Cur { int jj, n; };
            auto first = [&]() {
                Cur c{0, 0};
                while (p.kv_len[j0 + c.jj] == 0) ++c.jj;   // some block has keys
                return c;
            };
            auto next = [&](Cur c) {
                if (++c.n * BN >= p.kv_len[j0 + c.jj]) {
                    c.n = 0;
                    do ++c.jj; while (c.jj < nj && p.kv_len[j0 + c.jj] == 0);
                }
                return c;
            };
            auto load = [&](const CUtensorMap* maps, Cur c, uint8_t* dst, uint32_t full) {
                for (int ch = 0; ch < NCH; ++ch)
                    tma_load_4d(su32(dst + ch * CHUNK), &maps[j0 + c.jj], ch * 64, h, c.n * BN, b, full);
            };
            Cur vc = first(), kc = vc;
            // Q and K tile 0 first
            mbar_expect_tx(bar(B_Q), (NQT + 1) * TILE);
            for (int t = 0; t < NQT; ++t)
                for (int ch = 0; ch < NCH; ++ch)
                    tma_load_4d(su32(sQ + t * TILE + ch * CHUNK), &p.qmap[r], ch * 64, h, row_base + t * BM, b, bar(B_Q));
            load(p.kmap, kc, sK, bar(B_Q));
            kc = next(kc);
            int g = 0;
            bool ok = true;
            for (; g < total; ++g) {
                const int x = g & 1;
                if (g >= 1 && !(ok = wait_phase(bar(B_E + x), ((g - 1) >> 1) & 1, ctl))) break;
                if (g == total / 2) prefetch_next_cta<D, DIAG>(p);
                const bool has_k = g + 1 < total;
                mbar_expect_tx(bar(B_F + x), (has_k ? 2 : 1) * TILE);
                if (has_k) {
                    load(p.kmap, kc, sK + ((g + 1) & 1) * TILE, bar(B_F + x));
                    kc = next(kc);
                }
                load(p.vmap, vc, sV + x * TILE, bar(B_F + x));
                vc = next(vc);
            }
            if (!ok || *abort_flag) {
                // let every copy this thread issued land before smem is released
                drain_phase(bar(B_Q), 0);
                for (int k = g > 2 ? g - 2 : 0; k < g; ++k) drain_phase(bar(B_F + (k & 1)), (k >> 1) & 1);
            }
        }
        } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // The issuing thread stays inside tcgen05.mma until the tensor core
        // takes the instruction, and each commit or barrier wait after a
        // group of MMAs waits for that group to drain, so the waits and
        // commits are gathered into two gaps per position, where P must be
        // waited for in any case: P V(0, g) and Q K^T(0, g+1) go back to
        // back, so do P V(1, g) and Q K^T(1, g+1).
        if (lane == 0) {
            const uint32_t S[NQT] = {tmem, tmem + 128};
            const uint32_t O[NQT] = {tmem + 256, tmem + 256 + D};
            // Descriptors are built once; a k-step only adds an offset (in
            // 16-byte units) to the start-address field.  Stage buffers are
            // selected with (s ? x1 : x0), never by indexing an array.
            static_assert(NQT == 2 && NSK == 2 && kNSV == 2, "descriptor selection assumes 2 tiles and 2 stages");
            const uint64_t qd0 = sdesc(su32(sQ), 16, 1024), qd1 = sdesc(su32(sQ + TILE), 16, 1024);
            const uint64_t kd0 = sdesc(su32(sK), 16, 1024), kd1 = sdesc(su32(sK + TILE), 16, 1024);
            // V tile rows are keys (K dim), 64-wide d chunks CHUNK apart (N dim)
            const uint64_t vd0 = sdesc(su32(sV), CHUNK, 1024), vd1 = sdesc(su32(sV + TILE), CHUNK, 1024);
            const uint32_t idesc_qk = p.idesc_qk, idesc_pv = p.idesc_pv;
            auto issue_qk = [&](int t, int s) {
                const uint64_t a0 = t ? qd1 : qd0, b0 = s ? kd1 : kd0;
                const uint32_t d = t ? S[1] : S[0];
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t off = (uint64_t)(((ks & 3) * 32 + (ks >> 2) * CHUNK) >> 4);
                    mma_ss(d, a0 + off, b0 + off, idesc_qk, ks > 0);
                }
            };
            auto issue_pv = [&](int t, int s, bool acc) {
                const uint64_t b0 = s ? vd1 : vd0;
                const uint32_t d = t ? O[1] : O[0], a = t ? S[1] : S[0];
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    mma_ts(d, a + ks * 8, b0 + (uint64_t)(ks * 16 * 128 / 16), idesc_pv, (acc || ks > 0) ? 1u : 0u);
            };
            const int j0 = cta.j;
            auto tiles_of = [&](int jj) { return (p.kv_len[j0 + jj] + BN - 1) / BN; };
            // positions (key block jj, key tile n), empty blocks skipped; g
            // counts positions over the whole walk
            int jj = 0;
            while (tiles_of(jj) == 0) ++jj;       // some block has keys
            int nt = tiles_of(jj), n = 0;
            uint32_t g = 0;
            bool ok = wait_phase(bar(B_Q), 0, ctl);
            if (ok) {
                tc_fence_after();
                issue_qk(0, 0);
                tc_commit(bar(B_SF + 0));
                issue_qk(1, 0);
                tc_commit(bar(B_SF + 1));
                tc_commit(bar(B_E + 1));           // K tile 0 read (pair -1)
            }
            while (ok) {
                const int x = (int)(g & 1);
                // pair g: K tile g+1 (when there is one) and V tile g
                if (!(ok = wait_phase(bar(B_F + x), (g >> 1) & 1, ctl))) break;
                if (!(ok = wait_phase(bar(B_PF + 0), g & 1, ctl))) break;
                tc_fence_after();
                const bool last = n + 1 == nt;
                int jn = jj, nn = n + 1;
                if (last) {
                    nn = 0;
                    do ++jn; while (jn < nj && tiles_of(jn) == 0);
                }
                const bool more = jn < nj;
                // output done for a tile (the block's partial; folding, the
                // whole walk): its epilogue overlaps the next block's Q K^T
                const bool done = last && (!FOLD || !more);
                // folding, P V accumulates across the key blocks: only the
                // very first position starts O afresh
                const bool acc = FOLD ? g > 0 : n > 0;
                issue_pv(0, x, acc);
                if (done) tc_commit(bar(B_OD + 0));
                if (more) {
                    issue_qk(0, x ^ 1);
                    tc_commit(bar(B_SF + 0));
                }
                if (!(ok = wait_phase(bar(B_PF + 1), g & 1, ctl))) break;
                tc_fence_after();
                issue_pv(1, x, acc);
                if (done) tc_commit(bar(B_OD + 1));
                if (more) {
                    issue_qk(1, x ^ 1);
                    tc_commit(bar(B_SF + 1));
                }
                tc_commit(bar(B_E + x));           // K tile g+1 and V tile g read
                ++g;
                if (!more) break;
                if (last) nt = tiles_of(jn);
                jj = jn;
                n = nn;
            }
            tc_commit(bar(B_END));
            if (!ok) drain_phase(bar(B_END), 0);   // every issued MMA has finished
        }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2, q4 = warp & 3;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t St = tmem + t * 128 + lane_off;
        const uint32_t Ot = tmem + 256 + t * D + lane_off;
        const float c = p.c;
        bool ok = true;
        // one register of loop state: bit 0 the S/P phase (per key tile),
        // bit 1 the O-done phase (per block), bit 2 a key tile seen (folding),
        // bits 8.. the key block
        uint32_t st = 0;
        float m_used = 0.f, l = 0.f;          // folding: carried across the key blocks
        for (; (int)(st >> 8) < nj && ok; st += 256u) {
            int rem = p.kv_len[(DIAG ? cta_coords<DIAG>(p).j : 0) + (int)(st >> 8)];   // keys not yet seen
            if (rem == 0) {
                if (!FOLD) {
                    const Cta e = cta_coords<DIAG>(p);
                    write_empty_partial<D>(p, e.r, e.j + (int)(st >> 8), e.b, e.h, e.row_base);
                }
                continue;
            }
            if (!FOLD) m_used = l = 0.f;
            for (int n = 0; rem > 0; ++n, rem -= BN) {
                ok = __all_sync(0xffffffffu, wait_phase(bar(B_SF + t), st & 1, ctl));
                if (!ok) break;
                tc_fence_after();
                softmax_tile<D, P_BF16>(St, Ot, rem, n == 0 && !(st & 4u), c, m_used, l);
                mbar_arrive(bar(B_PF + t));
                st ^= 1u;
            }
            if (!ok) break;
            if (FOLD) st |= 4u;           // later blocks continue the running max and sum
            if (FOLD) {
                // the walk goes on into a later block with keys: no output yet
                bool later = false;
                for (int jj = (int)(st >> 8) + 1; jj < nj; ++jj) later |= p.kv_len[jj] > 0;
                if (later) continue;
            }
            // epilogue of block j: O / l and lse = ln(2) * (m + log2 l).  This
            // tile's "O done" barrier; the tile index is re-read from %tid
            // (volatile) and the address recomputed from the array's own
            // address, so that nothing derived from them stays live in the
            // key-tile loop, where the softmax needs every register.
            uint32_t tid_now;
            asm volatile("mov.u32 %0, %%tid.x;" : "=r"(tid_now));
            const uint32_t sbase = (su32(smem_raw) + 1023u) & ~1023u;
            // the thread's place, re-derived from %tid as well
            const int te = (int)(tid_now >> 7), we = (int)(tid_now >> 5), le = (int)(tid_now & 31);
            const uint32_t od_bar = sbase + (uint32_t)(BARS + (B_OD + te) * 8);
            ok = __all_sync(0xffffffffu, wait_phase(od_bar, (st >> 1) & 1, ctl));
            st ^= 2u;
            if (!ok) break;
            tc_fence_after();
            const float inv = 1.f / l;
            const Cta e = cta_coords<DIAG>(p);
            const int j = e.j + (int)(st >> 8);
            const int jc = (DIAG || FOLD) ? 0 : j;     // the output map's key-block coordinate
            const int eb = dtype_bytes(p.o_dt);
            const int rt = (int)(tid_now & 127);      // row within the tile
            const int row = e.row_base + te * BM + rt;
            if (p.lse.ptr && row < p.q_len[e.r])
                p.lse.ptr[e.r * p.lse.stride_q + j * p.lse.stride_kv + e.b * p.lse.stride_b + e.h * p.lse.stride_h +
                          p.q_row0[e.r] + row] = (m_used + log2f(l)) * 0.69314718055994531f;
            // The output goes through shared memory (per 128 bytes of d, rows
            // of 128 bytes, 16-byte chunks swizzled by row mod 8) and a TMA
            // store of each warp's 32 rows; rows past the block's length are
            // clipped by the output map.  The warp's own slot takes one
            // 128-byte column box at a time (the Q, K and V buffers are still
            // in use by the next block); the O row comes from TMEM in one
            // round trip.
            const uint32_t slot = sbase + (uint32_t)((NQT + NSK + NSV) * TILE + we * kSlot);
            const uint32_t myrow = slot + (uint32_t)le * 128u;
            const int grow = e.row_base + te * BM + (rt & ~31);
            uint32_t x[D];
            if constexpr (D == 128) tmem_ld128(Ot, x); else tmem_ld64(Ot, x);
            auto open_slot = [&]() {
                if (le == 0) bulk_wait_read();     // the slot's last store has read it
                __syncwarp();
            };
            auto store_box = [&](int bx) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (le == 0) {
                    tma_store_5d(&p.omap[e.r], slot, bx * (128 / eb), e.h, grow, e.b, jc);
                    bulk_commit();
                }
            };
            if (p.o_dt == DIT_F32) {
#pragma unroll
                for (int bx = 0; bx < D / 32; ++bx) {
                    open_slot();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int i = bx * 32 + 4 * k;
                        st_shared16(myrow + (uint32_t)((k ^ (le & 7)) << 4), __float_as_uint(__uint_as_float(x[i]) * inv),
                                    __float_as_uint(__uint_as_float(x[i + 1]) * inv),
                                    __float_as_uint(__uint_as_float(x[i + 2]) * inv),
                                    __float_as_uint(__uint_as_float(x[i + 3]) * inv));
                    }
                    store_box(bx);
                }
            } else {
#pragma unroll
                for (int bx = 0; bx < D / 64; ++bx) {
                    open_slot();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int i = bx * 64 + 8 * k;
                        uint32_t w[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            w[q] = pack2(__uint_as_float(x[i + 2 * q]) * inv, __uint_as_float(x[i + 2 * q + 1]) * inv,
                                         p.o_dt);
                        st_shared16(myrow + (uint32_t)((k ^ (le & 7)) << 4), w[0], w[1], w[2], w[3]);
                    }
                    store_box(bx);
                }
            }
        }
        // the shared-memory sources must stay until the copies have read
        // them; the global writes complete with the grid, before any
        // dependent kernel passes its griddepcontrol.wait
        if (lane == 0) bulk_wait_read();
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ---- host side --------------------------------------------------------------
std::atomic<void*> g_encode{nullptr};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    void* f = g_encode.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return nullptr;
        g_encode.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// 4-D map over [B][rows][H][D] (innermost first: d, h, row, b) with a
// 64 x 1 x 128 x 1 box and 128-byte swizzle; rows past `rows` read as 0.
dit_status make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, dit_dtype dt,
                    int D, int H, int rows, int B, int64_t sh, int64_t ss, int64_t sb) {
    if (rows < 1) rows = 1;     // never read: the kernel skips empty blocks
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    const int64_t sbb = B > 1 ? sb : (int64_t)rows * ss;   // unused when B == 1
    const cuuint64_t strides[3] = {(cuuint64_t)(sh * 2), (cuuint64_t)(ss * 2), (cuuint64_t)(sbb * 2)};
    const cuuint32_t box[4] = {64, 1, BM, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = enc(m, dt == DIT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                       const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return fail(DIT_ERR_INVALID_ARG, "attention: tensor map rejected (CUresult %d)", (int)res);
    return DIT_OK;
}

// 5-D map over the output view of one query block: (d, h, row, b, key
// block), a box of 128 bytes of d x 1 x 32 rows x 1 x 1 (one warp's rows),
// 128-byte swizzle.  Its
// extents are the block's own (rows = the block's query rows), so a store
// of a ragged last tile writes no row past the block.  Dimensions of extent
// 1 get the span of the dimensions inside them as stride; a zero stride on
// a longer dimension would send two rows to one address and is refused.
dit_status make_omap(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, void* base, dit_dtype dt, int D,
                     int H, int rows, int B, int nj, int64_t sh, int64_t ss, int64_t sb, int64_t sj) {
    const int eb = dtype_bytes(dt);
    if (rows < 1) rows = 1;     // never stored: the kernel skips empty blocks
    const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B, (cuuint64_t)nj};
    const int64_t st[4] = {sh, ss, sb, sj};
    cuuint64_t strides[4];
    uint64_t span = (uint64_t)D * eb;
    for (int i = 0; i < 4; ++i) {
        if (dims[i + 1] == 1) {
            strides[i] = span;
        } else {
            if (st[i] == 0) return fail(DIT_ERR_INVALID_ARG, "attention: zero output stride on a dimension longer than 1");
            strides[i] = (cuuint64_t)st[i] * eb;
        }
        span = strides[i] * dims[i + 1];
    }
    const cuuint32_t box[5] = {(cuuint32_t)(128 / eb), 1, 32, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType ty = dt == DIT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dt == DIT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult res = enc(m, ty, 5, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS)
        return fail(DIT_ERR_INVALID_ARG, "attention: output tensor map rejected (CUresult %d)", (int)res);
    return DIT_OK;
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp32 accumulation.
uint32_t make_idesc(bool bf16, bool b_mn_major, int N, int M) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int D, bool PB>
dit_status launch_kernel(const TcParams& prm, dim3 grid, cudaStream_t st) {
    int smem = smem_bytes<D>();
    if (smem < 116 * 1024) smem = 116 * 1024;   // one CTA per SM: it owns all 512 TMEM columns
    auto kernel = prm.diag ? attn_tc_kernel<D, PB, true, false>
                           : (prm.fold ? attn_tc_kernel<D, PB, false, true> : attn_tc_kernel<D, PB, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "attention: %s", cudaGetErrorString(e));
    e = launch_pdl(kernel, grid, dim3(NTHREADS), (size_t)smem, st, prm);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "attention: launch failed: %s", cudaGetErrorString(e));
    return check_launch("dit_attn_partial(tcgen05)");
}

}  // namespace

dit_status launch_attn_tc(const AttnArgs& a, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return fail(DIT_ERR_CUDA, "attention: cuTensorMapEncodeTiled unavailable");
    TcParams params;                // kernel parameter block (~4.4 KB, on the stack)
    memset(&params, 0, sizeof(params));
    TcParams* prm = &params;
    dit_status s = DIT_OK;
    int maxq = 0;
    for (int r = 0; r < a.n_q && s == DIT_OK; ++r) {
        prm->q_len[r] = a.q_len[r];
        if (a.q_len[r] > maxq) maxq = a.q_len[r];
        prm->q_row0[r] = a.q_row0[r];
        prm->o_row0[r] = a.o_row0[r];
        const char* base = static_cast<const char*>(a.q.ptr) + (r * a.q.stride_q + (int64_t)a.q_row0[r] * a.q.stride_s) * 2;
        s = make_map(enc, &prm->qmap[r], base, a.qk_dt, a.D, a.H, a.q_len[r], a.B, a.q.stride_h, a.q.stride_s,
                     a.q.stride_b);
        if (s == DIT_OK) {
            // with diag, query block r writes key block r's partial only
            char* ob = static_cast<char*>(a.o.ptr) +
                       (r * a.o.stride_q + (a.diag ? r * a.o.stride_kv : 0) +
                        ((int64_t)a.q_row0[r] + a.o_row0[r]) * a.o.stride_s) *
                           dtype_bytes(a.o_dt);
            s = make_omap(enc, &prm->omap[r], ob, a.o_dt, a.D, a.H, a.q_len[r], a.B, (a.diag || a.fold) ? 1 : a.n_kv,
                          a.o.stride_h, a.o.stride_s, a.o.stride_b, a.o.stride_kv);
        }
    }
    for (int j = 0; j < a.n_kv && s == DIT_OK; ++j) {
        prm->kv_len[j] = a.kv_len[j];
        const char* kb = static_cast<const char*>(a.k.ptr) + (j * a.k.stride_kv + (int64_t)a.kv_row0[j] * a.k.stride_s) * 2;
        const char* vb = static_cast<const char*>(a.v.ptr) + (j * a.v.stride_kv + (int64_t)a.kv_row0[j] * a.v.stride_s) * 2;
        s = make_map(enc, &prm->kmap[j], kb, a.qk_dt, a.D, a.H, a.kv_len[j], a.B, a.k.stride_h, a.k.stride_s,
                     a.k.stride_b);
        if (s == DIT_OK)
            s = make_map(enc, &prm->vmap[j], vb, a.v_dt, a.D, a.H, a.kv_len[j], a.B, a.v.stride_h, a.v.stride_s,
                         a.v.stride_b);
    }
    if (s == DIT_OK && maxq > 0) {
        prm->B = a.B; prm->n_q = a.n_q; prm->n_kv = a.n_kv; prm->diag = a.diag; prm->fold = a.fold; prm->nsm = num_sms();

        prm->c = a.scale * 1.4426950408889634f;
        prm->idesc_qk = make_idesc(a.qk_dt == DIT_BF16, false, BN, BM);
        prm->idesc_pv = make_idesc(a.v_dt == DIT_BF16, true, a.D, BM);
        prm->o = a.o; prm->o_dt = a.o_dt; prm->lse = a.lse; prm->status = a.status;
        // One CTA per (256 query rows, head, query block, batch) walks every
        // key block (with diag, its own block): measured on one GB300 against
        // one CTA per (query block, key block), 1153 against 1080 TFLOP/s at
        // 18 key tiles per block, 1369 against 1308 at 28, 1448 against 1437
        // at 148, and the same 1296 with a single key block.
        dim3 grid((maxq + NQT * BM - 1) / (NQT * BM), a.H, a.n_q * a.B);
        const bool pb = a.v_dt == DIT_BF16;
        if (grid.y > 65535 || grid.z > 65535) s = fail(DIT_ERR_UNSUPPORTED, "attention: grid too large");
        else if (a.D == 128)
            s = pb ? launch_kernel<128, true>(*prm, grid, st) : launch_kernel<128, false>(*prm, grid, st);
        else
            s = pb ? launch_kernel<64, true>(*prm, grid, st) : launch_kernel<64, false>(*prm, grid, st);
    }
    return s;
}

}  // namespace ditsp
