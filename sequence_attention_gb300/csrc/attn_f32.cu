// fp32 attention on CUDA cores, for float32 Q/K/V.  Tensor cores have no
// fp32 multiply at fp32 precision, so this path keeps every product and sum
// in fp32 (FFMA) and uses the accurate expf/logf, which keeps the result
// within about 1e-6 of exact for the head dims it serves.
//
// One thread (two for D = 128) owns one query row: the scaled q and the
// running output accumulator live in registers; 32-key K/V tiles are staged
// in shared memory and read as broadcasts.  Online softmax per tile:
// m' = max(m, tile max), l' = l*e^(m-m') + sum_t e^(s_t-m'),
// acc' = acc*e^(m-m') + sum_t e^(s_t-m') v_t.
#include <math.h>
#include <string.h>

#include "attn_common.cuh"

namespace ditsp {
namespace {

template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int DT = D > 64 ? 64 : D;   // d values per thread
    constexpr int TPR = D / DT;           // threads per row
    constexpr int ROWS = 128 / TPR;
    constexpr int KT = 32;                // keys per shared-memory tile
    __shared__ __align__(16) float ks[KT][D];
    __shared__ __align__(16) float vs[KT][D];

    const int z = blockIdx.z;
    const int b = z % a.B;
    // folding: z = (r, b) and the CTA walks every key block j in turn with
    // one running (m, l, acc) -- the ring's per-hop online-softmax merge
    const int j = a.fold ? 0 : (a.diag ? z / a.B : (z / a.B) % a.n_kv);
    const int r = a.fold ? z / a.B : (a.diag ? j : z / (a.B * a.n_kv));
    const int h = blockIdx.y;
    const int row0 = blockIdx.x * ROWS;
    const int qlen = a.q_len[r];
    if (row0 >= qlen) return;

    pdl_wait();
    const int tr = threadIdx.x / TPR, part = threadIdx.x % TPR;
    const int i = row0 + tr;
    const bool valid = i < qlen;

    const float* qp = static_cast<const float*>(a.q.ptr) + r * a.q.stride_q + b * a.q.stride_b +
                      ((long long)a.q_row0[r] + (valid ? i : 0)) * a.q.stride_s + h * a.q.stride_h + part * DT;
    float q[DT], acc[DT];
#pragma unroll
    for (int d = 0; d < DT; d += 4) {
        float4 x = valid ? *reinterpret_cast<const float4*>(qp + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        q[d] = x.x * a.scale; q[d + 1] = x.y * a.scale; q[d + 2] = x.z * a.scale; q[d + 3] = x.w * a.scale;
        acc[d] = acc[d + 1] = acc[d + 2] = acc[d + 3] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    const int j_end = a.fold ? a.n_kv : j + 1;
    for (int jb = j; jb < j_end; ++jb) {
    const int kvlen = a.kv_len[jb];
    const float* kb = static_cast<const float*>(a.k.ptr) + jb * a.k.stride_kv + b * a.k.stride_b + h * a.k.stride_h +
                      (long long)a.kv_row0[jb] * a.k.stride_s;
    const float* vb = static_cast<const float*>(a.v.ptr) + jb * a.v.stride_kv + b * a.v.stride_b + h * a.v.stride_h +
                      (long long)a.kv_row0[jb] * a.v.stride_s;

    for (int kt = 0; kt < kvlen; kt += KT) {
        __syncthreads();
        for (int e = threadIdx.x; e < KT * (D / 4); e += blockDim.x) {
            const int t = e / (D / 4), d4 = (e % (D / 4)) * 4;
            float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
            if (kt + t < kvlen) {
                kx = *reinterpret_cast<const float4*>(kb + (long long)(kt + t) * a.k.stride_s + d4);
                vx = *reinterpret_cast<const float4*>(vb + (long long)(kt + t) * a.v.stride_s + d4);
            }
            *reinterpret_cast<float4*>(&ks[t][d4]) = kx;
            *reinterpret_cast<float4*>(&vs[t][d4]) = vx;
        }
        __syncthreads();
        const int nk = min(KT, kvlen - kt);
        float s[KT];
        float tmax = -INFINITY;
#pragma unroll
        for (int t = 0; t < KT; ++t) {
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < DT; ++d) dot = fmaf(q[d], ks[t][part * DT + d], dot);
            if (TPR == 2) dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            s[t] = (t < nk) ? dot : -INFINITY;
            tmax = fmaxf(tmax, s[t]);
        }
        const float mnew = fmaxf(m, tmax);
        const float corr = expf(m - mnew);      // m = -inf on the first tile -> 0
        l *= corr;
#pragma unroll
        for (int d = 0; d < DT; ++d) acc[d] *= corr;
#pragma unroll
        for (int t = 0; t < KT; ++t) {
            const float p = (t < nk) ? expf(s[t] - mnew) : 0.f;
            l += p;
#pragma unroll
            for (int d = 0; d < DT; ++d) acc[d] = fmaf(p, vs[t][part * DT + d], acc[d]);
        }
        m = mnew;
    }
    }
    if (!valid) {
        pdl_trigger();
        return;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;          // l >= 1 once any key was seen
    float* op = static_cast<float*>(a.o.ptr) + r * a.o.stride_q + j * a.o.stride_kv + b * a.o.stride_b +
                ((long long)a.q_row0[r] + a.o_row0[r] + i) * a.o.stride_s + h * a.o.stride_h + part * DT;
#pragma unroll
    for (int d = 0; d < DT; d += 4)
        *reinterpret_cast<float4*>(op + d) = make_float4(acc[d] * inv, acc[d + 1] * inv, acc[d + 2] * inv, acc[d + 3] * inv);
    if (a.lse.ptr && part == 0)
        a.lse.ptr[r * a.lse.stride_q + j * a.lse.stride_kv + b * a.lse.stride_b + h * a.lse.stride_h + a.q_row0[r] + i] =
            l > 0.f ? m + logf(l) : -INFINITY;
    pdl_trigger();
}

}  // namespace

dit_status launch_attn_f32(const AttnArgs& a, cudaStream_t st) {
    int maxq = 0;
    for (int r = 0; r < a.n_q; ++r) maxq = a.q_len[r] > maxq ? a.q_len[r] : maxq;
    if (maxq == 0) return DIT_OK;
    const int rows = a.D == 128 ? 64 : 128;
    dim3 grid((maxq + rows - 1) / rows, a.H, ((a.diag || a.fold) ? a.n_q : a.n_q * a.n_kv) * a.B);
    if (grid.y > 65535 || grid.z > 65535) return fail(DIT_ERR_UNSUPPORTED, "attention: grid too large");
    cudaError_t e;
    switch (a.D) {
        case 16: e = launch_pdl(attn_f32_kernel<16>, grid, dim3(128), 0, st, a); break;
        case 32: e = launch_pdl(attn_f32_kernel<32>, grid, dim3(128), 0, st, a); break;
        case 64: e = launch_pdl(attn_f32_kernel<64>, grid, dim3(128), 0, st, a); break;
        case 128: e = launch_pdl(attn_f32_kernel<128>, grid, dim3(128), 0, st, a); break;
        default: return fail(DIT_ERR_UNSUPPORTED, "attention: fp32 path supports D in {16,32,64,128}");
    }
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "attention: launch failed: %s", cudaGetErrorString(e));
    return check_launch("dit_attn_partial(f32)");
}

}  // namespace ditsp
