// FP8 (e4m3) wire of the Ulysses exchange (cache-dit "Context Parallelism",
// Async FP8 Ulysses Attention: Q, V and the attention output O cross the
// all-to-all in float8, K stays 16-bit for the softmax's sake).
//
// Each (token, head) travels as one record of D + 16 bytes: the D e4m3 codes
// of x * (1/s), then s = amax/448 as a float32, then 12 zero bytes.  Every
// step that decides a code is an IEEE float32 operation with round to
// nearest even (amax, s = amax / 448, r = 1 / s, y = x * r, then the e4m3
// conversion with saturation), so a CPU float32 evaluation gives the same
// codes.  Decoding is code * s in float32, then one rounding to the
// destination type (and, in the receive preparation, the RoPE rotation of the
// float32 values before that rounding).
//
// The packs and the head -> seq unpack walk the same runs (Hl heads of one
// (plane, batch, row)) in the same destination orders as the 16-bit
// permutation kernels; a block decodes its runs into shared memory, each warp
// then covers its runs' heads with D/32 lanes per head, so the head's amax is
// a shuffle reduction inside an aligned group of lanes (32 values per lane;
// 16 when D = 16).  The seq -> head unpack takes one head-layout row per
// warp, a lane 8 values of one head at a time (fp8_unpack_rows_kernel).  The
// exchange between the pack and the unpack is the 16-bit exchange on records
// seen as (D + 16) / 2 words.
#include <cuda_fp8.h>
#include <string.h>

#include "convert.cuh"
#include "sp_index.cuh"

namespace ditsp {
namespace {

// The seq -> head decoding unpack is fp8_unpack_rows_kernel (below).
enum Fp8Mode { Q_PACK_S2H = 0, Q_PACK_H2S, DQ_UNPACK_H2S };

constexpr int kThreads = 256;

struct Fp8Args {
    dit_sp_layout L;
    int np;
    int lg;                        // log2 of the lanes that share one head
    const void* src[3];            // pack: planes (S2H) or head layout (H2S); unpack: wire
    const void* src2[3];           // paired streams (rows >= split), pack S2H only
    void* dst[3];                  // pack: wire; unpack: planes / output
    void* dst2[3];                 // paired streams, unpack H2S only
    int split;
    dit_dtype sdt;                 // 16/32-bit type of the pack's source
    dit_dtype ddt[3];              // 16/32-bit types of the unpack's destinations
    int* range_flag;
    long long nruns;
};

struct Fp8IO {
    const char* src;
    char* dst;
    int nslot;        // head slots (records) of the run
    int nreal;        // slots holding real heads; later slots (and padding rows) are zero
    int dt;           // the 16/32-bit side's dit_dtype
};

template <int MODE>
__device__ __forceinline__ Fp8IO fp8_io(const Fp8Args& A, int ri) {
    const dit_sp_layout& L = A.L;
    Run x;
    if (MODE == Q_PACK_S2H) x = decode_A(L, A.np, ri);
    else if (MODE == Q_PACK_H2S) x = decode_B(L, 1, ri);
    else x = decode_S(L, ri);
    const long long rec = L.D + 16;
    const bool pad_row = run_row(L, x) >= L.S;
    Fp8IO io;
    io.nslot = L.head_len[x.v];
    io.nreal = pad_row ? 0 : real_heads(L, x.v);
    bool second = false;
    if (MODE == Q_PACK_S2H) {
        io.dt = A.sdt;
        const long long so = io.nreal > 0 ? seq_offset(L, x, A.split, second) : 0;
        io.src = (const char*)(second ? A.src2[x.p] : A.src[x.p]) + so * dtype_bytes(A.sdt);
        io.dst = (char*)A.dst[0] + slots_A(L, A.np, x) * rec;
    } else if (MODE == Q_PACK_H2S) {
        io.dt = A.sdt;
        io.src = (const char*)A.src[0] + head_offset(L, x) * dtype_bytes(A.sdt);
        io.dst = (char*)A.dst[0] + slots_B(L, 1, x) * rec;
    } else {
        io.dt = A.ddt[0];
        io.src = (const char*)A.src[0] + slots_A(L, 1, x) * rec;
        const long long doff = io.nreal > 0 ? seq_offset(L, x, A.split, second) : 0;
        io.dst = (char*)(second ? A.dst2[0] : A.dst[0]) + doff * dtype_bytes(A.ddt[0]);
    }
    (void)ri;
    return io;
}

__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float2 from_e4m3x2(uint16_t v) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Quantize one lane's EPL values of a head with the head's reciprocal scale.
template <int EPL>
__device__ __forceinline__ void quant(const float (&x)[EPL], float r, uint4 (&out)[EPL / 16]) {
#pragma unroll
    for (int q = 0; q < EPL / 16; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = 16 * q + 4 * k;
            const uint32_t lo = to_e4m3x2(__fmul_rn(x[e], r), __fmul_rn(x[e + 1], r));
            const uint32_t hi = to_e4m3x2(__fmul_rn(x[e + 2], r), __fmul_rn(x[e + 3], r));
            w[k] = lo | (hi << 16);
        }
        out[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// EPL values held as raw 16-byte vectors of element size EB -> float32.
template <int EB, int EPL>
__device__ __forceinline__ void widen(const uint4 (&raw)[EPL * EB / 16], dit_dtype t, float (&x)[EPL]) {
#pragma unroll
    for (int v = 0; v < EPL / 8; ++v) {
        Vec8 f;
        load8(&raw[v * EB / 2], EB == 4 ? DIT_F32 : t, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[8 * v + k] = f.f[k];
    }
}

// Quantizing pack: source heads (16/32-bit) -> records.  A lane holds EPL
// consecutive values of a head, so D / EPL lanes share one head.
template <int MODE, int EB, int EPL>
__global__ void __launch_bounds__(kThreads, 3) fp8_pack_kernel(const __grid_constant__ Fp8Args A, int rpw) {
    constexpr int NV = EPL * EB / 16;        // 16-byte source vectors per lane and head
    constexpr int NU = EB == 4 ? 1 : 2;      // heads in flight per lane
    __shared__ Fp8IO ios[kThreads];
    const int rpb = rpw * (kThreads / 32);
    const long long r0 = (long long)blockIdx.x * rpb;
    const int nrun = (int)min((long long)rpb, A.nruns - r0);
    if ((int)threadIdx.x < nrun) ios[threadIdx.x] = fp8_io<MODE>(A, (int)(r0 + threadIdx.x));
    __syncthreads();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g0 = warp * rpw;
    const int gn = min(rpw, nrun - g0);
    if (gn <= 0) {
        pdl_trigger();
        return;
    }
    const int Hl = A.L.Hl, D = A.L.D, G = 1 << A.lg;
    const int units = gn * Hl;
    const int upw = 32 >> A.lg;                 // heads per warp per step
    const int c = lane & (G - 1);               // this lane's EPL-element slice of a head
    const int mine = lane >> A.lg;
    const dit_dtype sdt = A.sdt;
    // (run, head) of this lane's next unit, advanced by upw per unit
    int g = mine / Hl, hl = mine - (mine / Hl) * Hl;
    for (int base = 0; base < units; base += upw * NU) {   // warp-uniform trip count
        uint4 raw[NU][NV];
        int gh[NU];
#pragma unroll
        for (int b = 0; b < NU; ++b) {
            gh[b] = (g << 16) | hl;
            hl += upw;
            while (hl >= Hl) { hl -= Hl; ++g; }
        }
#pragma unroll
        for (int b = 0; b < NU; ++b) {
#pragma unroll
            for (int v = 0; v < NV; ++v) raw[b][v] = make_uint4(0, 0, 0, 0);
            const int u = base + b * upw + mine;
            if (u < units) {
                const int h = gh[b] & 0xffff;
                const Fp8IO& io = ios[g0 + (gh[b] >> 16)];
                if (h < io.nreal) {
                    const uint4* q = reinterpret_cast<const uint4*>(io.src + ((long long)h * D + c * EPL) * EB);
#pragma unroll
                    for (int v = 0; v < NV; ++v) raw[b][v] = q[v];
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NU; ++b) {
            const int u = base + b * upw + mine;
            float x[EPL];
            widen<EB, EPL>(raw[b], sdt, x);
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < EPL; ++k) amax = fmaxf(amax, fabsf(x[k]));
            for (int o = G >> 1; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (u < units && (gh[b] & 0xffff) < ios[g0 + (gh[b] >> 16)].nslot) {
                const float s = __fdiv_rn(amax, 448.f);
                const float r = s > 0.f ? __frcp_rn(s) : 0.f;
                char* rec = ios[g0 + (gh[b] >> 16)].dst + (long long)(gh[b] & 0xffff) * (D + 16);
                uint4 o[EPL / 16];
                quant<EPL>(x, r, o);
#pragma unroll
                for (int q = 0; q < EPL / 16; ++q) reinterpret_cast<uint4*>(rec + c * EPL)[q] = o[q];
                if (c == 0) *reinterpret_cast<uint4*>(rec + D) = make_uint4(__float_as_uint(s), 0u, 0u, 0u);
            }
        }
    }
    pdl_trigger();
}

// Dequantizing unpack, head -> seq: records -> sequence-layout heads
// (16/32-bit, real heads only).
template <int MODE, int EB, int EPL>
__global__ void __launch_bounds__(kThreads, 3) fp8_unpack_kernel(const __grid_constant__ Fp8Args A, int rpw) {
    constexpr int NC = EPL / 16;             // 16-byte code vectors per lane and head
    constexpr int NU = 4;                    // heads in flight per lane
    __shared__ Fp8IO ios[kThreads];
    const int rpb = rpw * (kThreads / 32);
    const long long r0 = (long long)blockIdx.x * rpb;
    const int nrun = (int)min((long long)rpb, A.nruns - r0);
    if ((int)threadIdx.x < nrun) ios[threadIdx.x] = fp8_io<MODE>(A, (int)(r0 + threadIdx.x));
    __syncthreads();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g0 = warp * rpw;
    const int gn = min(rpw, nrun - g0);
    if (gn <= 0) {
        pdl_trigger();
        return;
    }
    const int Hl = A.L.Hl, D = A.L.D, G = 1 << A.lg;
    const int units = gn * Hl;
    const int upw = 32 >> A.lg;
    const int c = lane & (G - 1);
    const int mine = lane >> A.lg;
    const bool check = A.range_flag != nullptr;
    bool overflow = false;
    int g = mine / Hl, hl = mine - (mine / Hl) * Hl;
    for (int base = mine; base < units; base += upw * NU) {
        uint4 code[NU][NC];
        float scale[NU];
        int gh[NU];
#pragma unroll
        for (int b = 0; b < NU; ++b) {
            gh[b] = (g << 16) | hl;
            hl += upw;
            while (hl >= Hl) { hl -= Hl; ++g; }
        }
#pragma unroll
        for (int b = 0; b < NU; ++b) {
#pragma unroll
            for (int q = 0; q < NC; ++q) code[b][q] = make_uint4(0, 0, 0, 0);
            scale[b] = 0.f;
            if (base + b * upw < units && (gh[b] & 0xffff) < ios[g0 + (gh[b] >> 16)].nslot) {
                const char* rec = ios[g0 + (gh[b] >> 16)].src + (long long)(gh[b] & 0xffff) * (D + 16);
#pragma unroll
                for (int q = 0; q < NC; ++q) code[b][q] = reinterpret_cast<const uint4*>(rec + c * EPL)[q];
                scale[b] = *reinterpret_cast<const float*>(rec + D);
            }
        }
#pragma unroll
        for (int b = 0; b < NU; ++b) {
            if (base + b * upw >= units) continue;
            const int h = gh[b] & 0xffff;
            const Fp8IO& io = ios[g0 + (gh[b] >> 16)];
            if (h >= io.nslot || (MODE == DQ_UNPACK_H2S && h >= io.nreal)) continue;
            const dit_dtype t = (dit_dtype)io.dt;
            char* dst = io.dst + ((long long)h * D + c * EPL) * dtype_bytes(t);
#pragma unroll
            for (int v = 0; v < EPL / 8; ++v) {          // 8 values at a time
                const uint32_t w0 = (&code[b][v >> 1].x)[(v & 1) * 2];
                const uint32_t w1 = (&code[b][v >> 1].x)[(v & 1) * 2 + 1];
                const uint32_t w[2] = {w0, w1};
                Vec8 y;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = from_e4m3x2((uint16_t)(w[k >> 1] >> (16 * (k & 1))));
                    y.f[2 * k] = __fmul_rn(f.x, scale[b]);
                    y.f[2 * k + 1] = __fmul_rn(f.y, scale[b]);
                }
                if (EB == 4) {
                    store8(dst + v * 32, DIT_F32, y);
                } else {
                    uint4 o = make_uint4(pack2(y.f[0], y.f[1], t), pack2(y.f[2], y.f[3], t),
                                         pack2(y.f[4], y.f[5], t), pack2(y.f[6], y.f[7], t));
                    if (check) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) overflow |= overflows16(y.f[e], t);
                    }
                    reinterpret_cast<uint4*>(dst)[v] = o;
                }
            }
        }
    }
    if (overflow) *A.range_flag = (int)DIT_ERR_RANGE;
    pdl_trigger();
}

// ---- seq -> head decoding unpack, one head-layout row per warp -----------
// As the three-call 16-bit unpack (direct.cu): lane v holds the record index
// of run v's first slot less head_off[v], so head h of the row is record
// rec(v(h)) + h; a lane takes 8 values of one head at a time (8 code bytes and
// the record's scale), decodes, rotates when asked (angle rows staged per
// warp) and stores them.  Same arithmetic as fp8_unpack_kernel.
constexpr int kRowThreads = 256;
constexpr int kRowItems = 8;
constexpr int kRowMaxRopeD = 256;

struct Fp8RowArgs {
    dit_sp_layout L;
    int np;
    const char* wire;
    char* head[3];
    dit_dtype ddt[3];
    int* range_flag;
    const float* rope_cos;
    const float* rope_sin;
    unsigned rope_planes;
    long long nrows;              // np * B * S_pad
    int cpr;                      // 8-value chunks per head-layout row (Hp * D / 8)
    int creal;                    // chunks of real heads (H * D / 8)
    FastDiv head_of;              // chunk -> head (D / 8 chunks a head)
    FastDiv group_of;             // head -> group when every group has Hl heads
    int even;
};

template <int DB, bool ROPE>
__global__ void __launch_bounds__(kRowThreads, 3) fp8_unpack_rows_kernel(const __grid_constant__ Fp8RowArgs A) {
    __shared__ float4 tab_sm[ROPE ? kRowThreads / 32 : 1][ROPE ? kRowMaxRopeD / 4 : 1];
    const dit_sp_layout& L = A.L;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long row = (long long)blockIdx.x * (kRowThreads / 32) + wib;
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
    const long long rec = L.D + 16;
    char* dst = A.head[p] + ((((long long)x.r * L.B + b) * L.S_cap + (t - L.ring_off[x.r])) * L.Hp) * L.D * DB;
    long long base = 0;        // lane v: run v's first record, less head_off[v]
    if (lane < L.U && lane < 32) {
        x.v = lane;
        base = slots_B(L, A.np, x) - L.head_off[lane];
    }
    const dit_dtype dt = A.ddt[p];
    const bool rot = ROPE && t < L.S && ((A.rope_planes >> p) & 1u);
    const int rlim = rot ? A.creal : 0;
    const bool check = A.range_flag != nullptr;
    bool overflow = false;
    const int q4 = L.D >> 3;
    if (ROPE && rot) {
        const float4* ct = reinterpret_cast<const float4*>(A.rope_cos + (long long)t * (L.D >> 1));
        const float4* sn = reinterpret_cast<const float4*>(A.rope_sin + (long long)t * (L.D >> 1));
        for (int j = lane; j < 2 * q4; j += 32) cp_async16(&tab_sm[wib][j], j < q4 ? ct + j : sn + (j - q4));
        cp_async_commit();
    }
    constexpr int NI = kRowItems;
    for (int c0 = 0; c0 < A.cpr; c0 += 32 * NI) {
        uint2 code[NI];
        float scale[NI];
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
            long long r0;
            if (L.U <= 32) {                                 // warp-uniform
                r0 = __shfl_sync(0xffffffffu, base, v);
            } else {
                Run y = x;
                y.v = v;
                r0 = slots_B(L, A.np, y) - L.head_off[v];
            }
            code[k] = make_uint2(0, 0);
            scale[k] = 0.f;
            if (c < A.cpr) {
                const char* r = A.wire + (r0 + h) * rec;
                code[k] = *reinterpret_cast<const uint2*>(r + (c - h * q4) * 8);
                scale[k] = *reinterpret_cast<const float*>(r + L.D);
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
            const uint32_t w[2] = {code[k].x, code[k].y};
            Vec8 y;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = from_e4m3x2((uint16_t)(w[e >> 1] >> (16 * (e & 1))));
                y.f[2 * e] = __fmul_rn(f.x, scale[k]);
                y.f[2 * e + 1] = __fmul_rn(f.y, scale[k]);
            }
            if (ROPE && c < rlim) {
                const int i4 = c - (int)fdiv((uint32_t)c, A.head_of) * q4;
                const float4 cc = tab_sm[wib][i4], ss = tab_sm[wib][q4 + i4];
                const float ca[4] = {cc.x, cc.y, cc.z, cc.w}, sa[4] = {ss.x, ss.y, ss.z, ss.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = y.f[2 * e], x1 = y.f[2 * e + 1];
                    y.f[2 * e] = fmaf(x0, ca[e], -(x1 * sa[e]));
                    y.f[2 * e + 1] = fmaf(x0, sa[e], x1 * ca[e]);
                }
            }
            char* d = dst + (long long)c * 8 * DB;
            if (DB == 4) {
                store8(d, DIT_F32, y);
            } else {
                if (check) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) overflow |= overflows16(y.f[e], dt);
                }
                *reinterpret_cast<uint4*>(d) = make_uint4(pack2(y.f[0], y.f[1], dt), pack2(y.f[2], y.f[3], dt),
                                                          pack2(y.f[4], y.f[5], dt), pack2(y.f[6], y.f[7], dt));
            }
        }
    }
    if (ROPE && rot) __syncwarp();
    if (overflow) *A.range_flag = (int)DIT_ERR_RANGE;
    pdl_trigger();
}

template <int DB, bool ROPE>
dit_status launch_rows(const Fp8RowArgs& a, cudaStream_t st, const char* who) {
    const long long blocks = (a.nrows + kRowThreads / 32 - 1) / (kRowThreads / 32);
    if (blocks >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: too many rows", who);
    cudaError_t e = launch_pdl(fp8_unpack_rows_kernel<DB, ROPE>, dim3((unsigned)blocks), dim3(kRowThreads), 0, st, a);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

template <typename K>
dit_status launch_fp8(K kernel, const Fp8Args& a, cudaStream_t st, const char* who) {
    if (a.nruns == 0) return DIT_OK;
    if (a.nruns >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: more than 2^31 runs", who);
    // 16 runs per warp (128 per block): measured against 1, 2, 4 and 8 on the
    // FLUX- and Wan-like shapes, the fastest at the Wan size (fewer runs per
    // block pay the per-block decode of run offsets more often).  When 16
    // would leave less than one wave of blocks (3 per SM), the fewest runs
    // per warp from 8 up whose grid fills at most 90 % of one wave: a grid
    // just over one wave leaves a tail of blocks that waits for the first
    // wave to drain.  FLUX-like Q and V pack (36,864 runs, 456 resident
    // blocks): 12 runs per warp, 384 blocks, 17.9 us; 8 (576 blocks) 19.2,
    // 10 (461) 22.3, 11 (419) 18.2, 16 (288) 19.9.
    const long long cap = 3LL * num_sms();
    int rpw = 16;
    if ((a.nruns + 127) / 128 < cap)
        for (rpw = 8; rpw < 16 && (a.nruns + 8LL * rpw - 1) / (8LL * rpw) > cap * 9 / 10; ++rpw) {
        }
    const long long blocks = (a.nruns + 8LL * rpw - 1) / (8LL * rpw);
    cudaError_t e = launch_pdl(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, a, rpw);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}

// lg = log2 of the lanes per head: D / 32 (D / 16 for D = 16)
dit_status check_fp8_shape(const dit_sp_layout* L, const char* who, int* lg) {
    const int D = L->D;
    if (D < 16 || D > 256 || (D & (D - 1)))
        return fail(DIT_ERR_UNSUPPORTED, "%s: the e4m3 wire needs D in {16, 32, 64, 128, 256}", who);
    const int epl = D == 16 ? 16 : 32;
    int g = 0;
    while ((epl << g) < D) ++g;
    *lg = g;
    return DIT_OK;
}

template <int EPL>
dit_status launch_unpack(const Fp8Args& a, bool wide, cudaStream_t st, const char* who) {
    return wide ? launch_fp8(fp8_unpack_kernel<DQ_UNPACK_H2S, 4, EPL>, a, st, who)
                : launch_fp8(fp8_unpack_kernel<DQ_UNPACK_H2S, 2, EPL>, a, st, who);
}

}  // namespace

dit_status fp8_pack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes, const void* const* src,
                    const void* const* src2, int split, dit_dtype src_dt, void* send, cudaStream_t st,
                    const char* who) {
    Fp8Args a;
    memset(&a, 0, sizeof(a));
    dit_status s = check_fp8_shape(L, who, &a.lg);
    if (s != DIT_OK) return s;
    a.L = *L;
    a.np = nplanes;
    for (int p = 0; p < nplanes; ++p) {
        a.src[p] = src ? src[p] : nullptr;
        a.src2[p] = src2 ? src2[p] : nullptr;
    }
    a.split = split;
    a.sdt = src_dt;
    a.dst[0] = send;
    a.nruns = (long long)nplanes * L->B * L->U * L->S_pad;
    const bool wide = dtype_bytes(src_dt) == 4;
    if (L->D == 16) {
        if (dir == DIT_SEQ_TO_HEAD)
            return wide ? launch_fp8(fp8_pack_kernel<Q_PACK_S2H, 4, 16>, a, st, who)
                        : launch_fp8(fp8_pack_kernel<Q_PACK_S2H, 2, 16>, a, st, who);
        return wide ? launch_fp8(fp8_pack_kernel<Q_PACK_H2S, 4, 16>, a, st, who)
                    : launch_fp8(fp8_pack_kernel<Q_PACK_H2S, 2, 16>, a, st, who);
    }
    if (dir == DIT_SEQ_TO_HEAD)
        return wide ? launch_fp8(fp8_pack_kernel<Q_PACK_S2H, 4, 32>, a, st, who)
                    : launch_fp8(fp8_pack_kernel<Q_PACK_S2H, 2, 32>, a, st, who);
    return wide ? launch_fp8(fp8_pack_kernel<Q_PACK_H2S, 4, 32>, a, st, who)
                : launch_fp8(fp8_pack_kernel<Q_PACK_H2S, 2, 32>, a, st, who);
}

dit_status fp8_unpack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes, const void* recv, void* const* dst,
                      void* const* dst2, int split, const dit_dtype* dst_dt, const float* cos_tab,
                      const float* sin_tab, unsigned rope_planes, int* range_flag, cudaStream_t st,
                      const char* who) {
    const int db = dtype_bytes(dst_dt[0]);
    if (dir == DIT_SEQ_TO_HEAD) {
        int lg;
        dit_status s = check_fp8_shape(L, who, &lg);
        if (s != DIT_OK) return s;
        for (int p = 1; p < nplanes; ++p)
            if (dtype_bytes(dst_dt[p]) != db)
                return fail(DIT_ERR_UNSUPPORTED, "%s: planes of one call need destination types of one size", who);
        if (L->U > 64) return fail(DIT_ERR_UNSUPPORTED, "%s: more than 64 Ulysses ranks", who);
        Fp8RowArgs a;
        memset(&a, 0, sizeof(a));
        a.L = *L;
        a.np = nplanes;
        a.wire = static_cast<const char*>(recv);
        for (int p = 0; p < nplanes; ++p) {
            a.head[p] = static_cast<char*>(dst[p]);
            a.ddt[p] = dst_dt[p];
        }
        a.range_flag = range_flag;
        a.rope_cos = cos_tab;
        a.rope_sin = sin_tab;
        a.rope_planes = rope_planes;
        a.nrows = (long long)nplanes * L->B * L->S_pad;
        a.cpr = (int)(((long long)L->Hp * L->D) >> 3);
        a.creal = (int)(((long long)L->H * L->D) >> 3);
        a.head_of = make_fastdiv((uint32_t)(L->D >> 3));
        a.even = 1;
        for (int v = 0; v < L->U; ++v) a.even &= L->head_len[v] == L->Hl && L->head_off[v] == v * L->Hl;
        a.group_of = make_fastdiv((uint32_t)(L->Hl > 0 ? L->Hl : 1));
        if (a.nrows == 0) return DIT_OK;
        if (rope_planes) return db == 4 ? launch_rows<4, true>(a, st, who) : launch_rows<2, true>(a, st, who);
        return db == 4 ? launch_rows<4, false>(a, st, who) : launch_rows<2, false>(a, st, who);
    }
    Fp8Args a;
    memset(&a, 0, sizeof(a));
    dit_status s = check_fp8_shape(L, who, &a.lg);
    if (s != DIT_OK) return s;
    a.L = *L;
    a.np = nplanes;
    a.src[0] = recv;
    for (int p = 0; p < nplanes; ++p) {
        a.dst[p] = dst[p];
        a.dst2[p] = dst2 ? dst2[p] : nullptr;
        a.ddt[p] = dst_dt[p];
        if (dtype_bytes(dst_dt[p]) != db)
            return fail(DIT_ERR_UNSUPPORTED, "%s: planes of one call need destination types of one size", who);
    }
    a.split = split;
    a.range_flag = range_flag;
    a.nruns = (long long)nplanes * L->B * L->U * L->S;
    if (L->D == 16) return launch_unpack<16>(a, db == 4, st, who);
    return launch_unpack<32>(a, db == 4, st, who);
}

}  // namespace ditsp
