// Bandwidth-bound elementwise steps: the classifier-free guidance combine and
// the log-sum-exp merge of ring partials.
//
// CFG (edge-dit.cpp "Parallel execution", classifier-free guidance):
//   p = p_uncond + g * (p_cond - p_uncond), evaluated literally in fp32 as
//   fma(g, p_cond - p_uncond, p_uncond) and fused with the cast to the output
//   type.  g = 0 gives p_uncond exactly; for g = 1 the formula reduces to
//   p_cond, which is returned as is (fp32 rounding of p_cond - p_uncond could
//   otherwise move it when the two differ by many binades).
// Merge (SGLang Diffusion "Parallelism Overview", What happens to the shapes /
// Constraints: the ring's online-softmax merge over same-head, different-row
// partials):  lse = M + ln sum_j exp(lse_j - M),  O = sum_j exp(lse_j - lse) O_j
// (evaluated as sum_j (e_j / sum e) O_j with e_j = exp(lse_j - M)).
#include <math.h>
#include <string.h>

#include "common.cuh"

namespace ditsp {
namespace {

// ---------------------------------------------------------------------------
// CFG: a one-shot grid (no grid-stride loop); each thread combines four
// 8-element vectors spaced one block apart (coalesced), issuing all eight
// 16-byte loads before any arithmetic.
constexpr int kCfgThreads = 256;
constexpr int kCfgVecs = 4;

template <int IB>   // input element bytes
__global__ void __launch_bounds__(kCfgThreads) cfg_vec_kernel(const char* __restrict__ pred, dit_dtype in_dt,
                                                              long long nvec, long long N, float g,
                                                              char* __restrict__ out, dit_dtype out_dt) {
    const long long base = (long long)blockIdx.x * (kCfgThreads * kCfgVecs) + threadIdx.x;
    const char* cond = pred + N * IB;
    pdl_wait();
    uint4 ru[kCfgVecs][IB / 2], rc[kCfgVecs][IB / 2];
#pragma unroll
    for (int k = 0; k < kCfgVecs; ++k) {
        const long long v = base + (long long)k * kCfgThreads;
        if (v < nvec) {
#pragma unroll
            for (int h = 0; h < IB / 2; ++h) {
                ru[k][h] = reinterpret_cast<const uint4*>(pred + v * 8 * IB)[h];
                rc[k][h] = reinterpret_cast<const uint4*>(cond + v * 8 * IB)[h];
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kCfgVecs; ++k) {
        const long long v = base + (long long)k * kCfgThreads;
        if (v < nvec) {
            Vec8 u, c, p;
            load8(&ru[k][0], in_dt, u);
            load8(&rc[k][0], in_dt, c);
            if (g == 1.0f) {
                p = c;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) p.f[e] = fmaf(g, c.f[e] - u.f[e], u.f[e]);
            }
            store8(out + v * 8 * dtype_bytes(out_dt), out_dt, p);
        }
    }
    pdl_trigger();
}

__device__ __forceinline__ float load1(const char* p, dit_dtype t, long long i) {
    if (t == DIT_F32) return reinterpret_cast<const float*>(p)[i];
    if (t == DIT_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ void store1(char* p, dit_dtype t, long long i, float x) {
    if (t == DIT_F32) reinterpret_cast<float*>(p)[i] = x;
    else if (t == DIT_BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<__half*>(p)[i] = __float2half_rn(x);
}

// Scalar tail / unaligned-length path.
__global__ void cfg_scalar_kernel(const char* __restrict__ pred, dit_dtype in_dt, long long begin,
                                  long long N, float g, char* __restrict__ out, dit_dtype out_dt) {
    pdl_wait();
    for (long long i = begin + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < N;
         i += (long long)gridDim.x * blockDim.x) {
        const float u = load1(pred, in_dt, i), c = load1(pred, in_dt, N + i);
        store1(out, out_dt, i, g == 1.0f ? c : fmaf(g, c - u, u));
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Merge arguments: grid y is (r, b); x covers rows * heads * D/8 chunks of the
// longest block.
struct MergeArgs {
    int B, H, D, n_parts;
    int n_q_b;                  // n_q * B (grid y)
    int q_len[DIT_MAX_R];
    dit_view parts;
    dit_dtype parts_dt;
    dit_lse_view lse_parts;
    dit_view out;
    dit_dtype out_dt;
    dit_lse_view lse_out;
};

// The SFU's base-2 exponential and reciprocal (relative errors about 2^-22
// and 2^-23): ex2(-inf) = 0, so an empty partial gets weight 0.
__device__ __forceinline__ float sfu_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sfu_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge, chunk-per-thread form: thread t of block (x, r*B + b) takes CPT
// 8-element chunks of unit u = (row i, head h), D / 8 / CPT chunks apart (so
// each load instruction of a warp still covers whole 128-byte segments) --
// the same weights for all of them -- and SLOTS such groups spaced one
// block apart.
// Every load of a thread -- the NP log-sum-exp values and the NP partial
// chunks of each of its slots -- is issued before any arithmetic, so one
// memory round trip covers all of them (the lanes of one unit read the same
// log-sum-exp words, served by one transaction).  Each thread forms its
// unit's weights itself as w_j = e_j / sum_j e_j with e_j = 2^((lse_j - M)
// log2 e): NP SFU exponentials and one SFU reciprocal per 8 * CPT outputs
// (relative error of a weight below 1e-6, far inside the merge's fp32
// bound), and the merged log-sum-exp (an accurate logarithm) only when it is
// asked for.  Index decoding is 32-bit, with divisions by the launch's fixed
// row and head sizes done as multiply-shifts.  A thread keeps 64 (16-bit
// parts) or 128 bytes of partials in flight.  Units run h-fastest within a
// row and chunks c-fastest within a head, so the block's loads and stores
// cover whole contiguous rows.
template <int NP, int SLOTS, int PB, int CPT>
__global__ void __launch_bounds__(256) merge_chunks_kernel(const __grid_constant__ MergeArgs a, FastDiv per_row,
                                                           FastDiv groups) {
    const int r = blockIdx.y / a.B, b = blockIdx.y % a.B;
    const uint32_t total = (uint32_t)a.q_len[r] * per_row.d;
    const uint32_t t0 = blockIdx.x * (blockDim.x * SLOTS) + threadIdx.x;
    const char* pp = static_cast<const char*>(a.parts.ptr);
    const dit_dtype pdt = a.parts_dt;
    const int cstride = (int)groups.d;   // chunks between a thread's CPT chunks (D / 8 / CPT)
    long long base[SLOTS];
    int lrow[SLOTS];           // row i of the slot's unit (-1: none)
    int lh[SLOTS], lc[SLOTS];  // head, first chunk (lc == 0: the thread writes the merged lse)
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        const uint32_t t = t0 + (uint32_t)k * blockDim.x;
        lrow[k] = -1;
        if (t < total) {
            const uint32_t i = fdiv(t, per_row);
            const uint32_t rem = t - i * per_row.d;
            const uint32_t h = fdiv(rem, groups);
            lrow[k] = (int)i;
            lh[k] = (int)h;
            lc[k] = (int)(rem - h * groups.d);          // chunks lc, lc + chunks/CPT, ...
            base[k] = r * a.parts.stride_q + b * a.parts.stride_b + (long long)i * a.parts.stride_s +
                      (long long)h * a.parts.stride_h + lc[k] * 8;
        }
    }
    pdl_wait();
    float lj[SLOTS][NP];
    uint4 raw[SLOTS][NP][CPT][PB / 2];
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        if (lrow[k] < 0) continue;
        const float* lp = a.lse_parts.ptr + r * a.lse_parts.stride_q + b * a.lse_parts.stride_b +
                          lh[k] * a.lse_parts.stride_h + lrow[k];
#pragma unroll
        for (int j = 0; j < NP; ++j) lj[k][j] = lp[j * a.lse_parts.stride_kv];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const uint4* q = reinterpret_cast<const uint4*>(pp + (base[k] + j * a.parts.stride_kv) * PB);
#pragma unroll
            for (int c = 0; c < CPT; ++c)
#pragma unroll
                for (int h = 0; h < PB / 2; ++h) raw[k][j][c][h] = q[c * cstride * (PB / 2) + h];
        }
    }
    char* op = static_cast<char*>(a.out.ptr);
    const int ob = dtype_bytes(a.out_dt);
    constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        if (lrow[k] < 0) continue;
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < NP; ++j) M = fmaxf(M, lj[k][j]);
        Vec8 acc[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[c].f[e] = 0.f;
        float lse = -INFINITY;
        if (M != -INFINITY) {
            float ej[NP];
            float sum = 0.f;
            const float mb = M * kLog2e;
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                ej[j] = sfu_ex2(fmaf(lj[k][j], kLog2e, -mb));    // 2^((lse_j - M) log2 e); -inf -> 0
                sum += ej[j];
            }
            const float inv = sfu_rcp(sum);                       // sum >= 1 (the largest part gives ~1)
            if (a.lse_out.ptr && lc[k] == 0) lse = M + logf(sum);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const float w = ej[j] * inv;
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    Vec8 o;
                    load8(&raw[k][j][c][0], pdt, o);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[c].f[e] = fmaf(w, o.f[e], acc[c].f[e]);
                }
            }
        }
        const long long off = r * a.out.stride_q + b * a.out.stride_b + (long long)lrow[k] * a.out.stride_s +
                              lh[k] * a.out.stride_h + lc[k] * 8;
#pragma unroll
        for (int c = 0; c < CPT; ++c) store8(op + (off + (long long)c * cstride * 8) * ob, a.out_dt, acc[c]);
        if (a.lse_out.ptr && lc[k] == 0)
            a.lse_out.ptr[r * a.lse_out.stride_q + b * a.lse_out.stride_b + lh[k] * a.lse_out.stride_h + lrow[k]] =
                lse;
    }
    pdl_trigger();
}

template <int NP, int PB>
cudaError_t launch_merge_chunks(const MergeArgs& a, long long work, cudaStream_t st) {
    const int chunks = a.D / 8;
    // two chunks per thread (one set of weights for 16 outputs) for three or
    // four 16-bit parts, when the head's chunk count is even: Wan-like R = 4
    // on f16 partials 540 against 627 us.  With two parts the weights cost
    // less than the second slot's independent loads gain (FLUX-1008 15.0
    // against 16.1 us, Qwen 40.2 against 42.1), and fp32 parts need the
    // registers.
    constexpr bool two = NP >= 3 && NP * PB <= 8;
    if (two && chunks % 2 == 0) {
        constexpr int CPT = two ? 2 : 1;
        constexpr int SLOTS = NP * CPT >= 4 ? 1 : 4 / (NP * CPT);
        const long long per_block = 256LL * SLOTS * CPT;
        const dim3 grid((unsigned)((work + per_block - 1) / per_block), (unsigned)a.n_q_b);
        const FastDiv per_row = make_fastdiv((uint32_t)(a.H * (chunks / CPT))), groups = make_fastdiv((uint32_t)(chunks / CPT));
        return launch_pdl(merge_chunks_kernel<NP, SLOTS, PB, CPT>, grid, dim3(256), 0, st, a, per_row, groups);
    }
    constexpr int SLOTS = NP >= 4 ? 1 : 4 / NP;
    const long long per_block = 256LL * SLOTS;
    const dim3 grid((unsigned)((work + per_block - 1) / per_block), (unsigned)a.n_q_b);
    const FastDiv per_row = make_fastdiv((uint32_t)(a.H * chunks)), groups = make_fastdiv((uint32_t)chunks);
    return launch_pdl(merge_chunks_kernel<NP, SLOTS, PB, 1>, grid, dim3(256), 0, st, a, per_row, groups);
}

template <int PB>
cudaError_t launch_merge(const MergeArgs& a, long long work, cudaStream_t st) {
    switch (a.n_parts) {
        case 1: return launch_merge_chunks<1, PB>(a, work, st);
        case 2: return launch_merge_chunks<2, PB>(a, work, st);
        case 3: return launch_merge_chunks<3, PB>(a, work, st);
        case 4: return launch_merge_chunks<4, PB>(a, work, st);
        case 5: return launch_merge_chunks<5, PB>(a, work, st);
        case 6: return launch_merge_chunks<6, PB>(a, work, st);
        case 7: return launch_merge_chunks<7, PB>(a, work, st);
        default: return launch_merge_chunks<8, PB>(a, work, st);
    }
}

}  // namespace
}  // namespace ditsp

using namespace ditsp;

extern "C" dit_status dit_cfg_combine(const void* pred, dit_dtype in_dt, int64_t N, float g, void* out,
                                      dit_dtype out_dt, void* stream) {
    NvtxRange nvtx_range("dit_cfg_combine");
    const char* who = "dit_cfg_combine";
    if (!dtype_ok(in_dt) || !dtype_ok(out_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (N < 0) return fail(DIT_ERR_INVALID_ARG, "%s: N < 0", who);
    if (N == 0) return DIT_OK;
    if (!pred || !out || !aligned16(pred) || !aligned16(out))
        return fail(DIT_ERR_INVALID_ARG, "%s: pred/out NULL or not 16-byte aligned", who);
    const char* pb = static_cast<const char*>(pred);
    const char* pe = pb + 2 * N * dtype_bytes(in_dt);
    const char* ob = static_cast<const char*>(out);
    const char* oe = ob + N * dtype_bytes(out_dt);
    if (ob < pe && pb < oe) return fail(DIT_ERR_INVALID_ARG, "%s: out overlaps pred", who);
    cudaStream_t st = (cudaStream_t)stream;
    // The vector path needs the conditional half 16-byte aligned too.
    const bool vec_ok = ((N * dtype_bytes(in_dt)) % 16) == 0;
    long long done = 0;
    if (vec_ok) {
        const long long nvec = N / 8;
        if (nvec > 0) {
            const long long blocks = (nvec + kCfgThreads * kCfgVecs - 1) / (kCfgThreads * kCfgVecs);
            cudaError_t e = launch_pdl(in_dt == DIT_F32 ? cfg_vec_kernel<4> : cfg_vec_kernel<2>, dim3((unsigned)blocks),
                                       dim3(kCfgThreads), 0, st, pb, in_dt, nvec, N, g, static_cast<char*>(out),
                                       out_dt);
            if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
            dit_status s = check_launch(who);
            if (s != DIT_OK) return s;
        }
        done = nvec * 8;
    }
    if (done < N) {
        const long long rest = N - done;
        long long blocks = (rest + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        cudaError_t e = launch_pdl(cfg_scalar_kernel, dim3((unsigned)blocks), dim3(256), 0, st, pb, in_dt, done, N, g,
                                   static_cast<char*>(out), out_dt);
        if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
        return check_launch(who);
    }
    return DIT_OK;
}

extern "C" dit_status dit_attn_merge_lse(int B, int H, int D, int n_q, const int* q_len, int n_parts,
                                         dit_view parts, dit_dtype parts_dt, dit_lse_view lse_parts,
                                         dit_view out, dit_dtype out_dt, dit_lse_view lse_out,
                                         void* stream) {
    NvtxRange nvtx_range("dit_attn_merge_lse");
    const char* who = "dit_attn_merge_lse";
    if (B < 1 || H < 1 || D < 8 || D % 8 != 0)
        return fail(DIT_ERR_INVALID_ARG, "%s: need B,H >= 1 and D a positive multiple of 8", who);
    if (n_q < 1 || n_q > DIT_MAX_R || !q_len || n_parts < 1 || n_parts > DIT_MAX_R)
        return fail(DIT_ERR_INVALID_ARG, "%s: need 1 <= n_q, n_parts <= %d", who, DIT_MAX_R);
    if (!dtype_ok(parts_dt) || !dtype_ok(out_dt)) return fail(DIT_ERR_INVALID_ARG, "%s: bad dtype", who);
    const int64_t pstr[] = {parts.stride_q, parts.stride_kv, parts.stride_b, parts.stride_s, parts.stride_h};
    const int64_t ostr[] = {out.stride_q, out.stride_b, out.stride_s, out.stride_h};
    for (int64_t s : pstr)
        if ((s * dtype_bytes(parts_dt)) % 16) return fail(DIT_ERR_INVALID_ARG, "%s: parts strides not 16-byte multiples", who);
    for (int64_t s : ostr)
        if ((s * dtype_bytes(out_dt)) % 16) return fail(DIT_ERR_INVALID_ARG, "%s: out strides not 16-byte multiples", who);
    MergeArgs a;
    memset(&a, 0, sizeof(a));
    a.B = B; a.H = H; a.D = D; a.n_parts = n_parts;
    int maxq = 0;
    for (int r = 0; r < n_q; ++r) {
        if (q_len[r] < 0) return fail(DIT_ERR_INVALID_ARG, "%s: negative q_len", who);
        a.q_len[r] = q_len[r];
        if (q_len[r] > maxq) maxq = q_len[r];
    }
    // no rows: nothing is read or written, and the (empty) buffers may be NULL
    if (maxq == 0) return DIT_OK;
    if (!parts.ptr || !out.ptr || !lse_parts.ptr || !aligned16(parts.ptr) || !aligned16(out.ptr))
        return fail(DIT_ERR_INVALID_ARG, "%s: NULL or misaligned pointer", who);
    a.parts = parts; a.parts_dt = parts_dt; a.lse_parts = lse_parts;
    a.out = out; a.out_dt = out_dt; a.lse_out = lse_out;
    if ((long long)n_q * B > 65535) return fail(DIT_ERR_UNSUPPORTED, "%s: n_q * B too large", who);
    a.n_q_b = n_q * B;
    const long long work = (long long)maxq * H * (D / 8);      // chunks of the longest block
    // 32-bit index decoding in the kernel: every block's chunk count, and the
    // grid's last chunk index, below 2^31
    if (work + 256LL * 4 >= (1LL << 31)) return fail(DIT_ERR_UNSUPPORTED, "%s: 2^31 or more chunks per block", who);
    const cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = parts_dt == DIT_F32 ? launch_merge<4>(a, work, st) : launch_merge<2>(a, work, st);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    return check_launch(who);
}
