/*
 * usp_step.c -- one sequence-parallel attention step and a CFG combine run
 * from plain C through the ditsp.h ABI, on device buffers from cudaMalloc.
 *
 *   usp_step <dir> S H D U R
 *
 * Reads <dir>/q.bin, k.bin, v.bin (bf16 [1][S][H][D]) and pred.bin (bf16
 * [2][N]); writes <dir>/out.bin (bf16 [1][S][H][D]) and cfg.bin (bf16 [N]).
 * The step is the three-call Ulysses exchange a multi-GPU build would keep:
 * seq->head pack, exchange, unpack (V to f16); every ring partial in one
 * attention call; the log-sum-exp merge; head->seq pack, exchange, unpack.
 * Prints "ok" and the device status word, or the failing call and its error.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ditsp.h"

#define CK(call)                                                                        \
    do {                                                                                \
        dit_status s_ = (call);                                                         \
        if (s_ != DIT_OK) {                                                             \
            printf("FAIL %s: %s (%s)\n", #call, dit_status_string(s_), dit_last_error()); \
            return 1;                                                                   \
        }                                                                               \
    } while (0)
#define CU(call)                                                                        \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess) {                                                        \
            printf("FAIL %s: %s\n", #call, cudaGetErrorString(e_));                     \
            return 1;                                                                   \
        }                                                                               \
    } while (0)

static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[1024];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) return NULL;
    void* p = malloc(bytes);
    size_t n = p ? fread(p, 1, bytes, f) : 0;
    fclose(f);
    if (n != bytes) {
        free(p);
        return NULL;
    }
    return p;
}

static int write_file(const char* dir, const char* name, const void* p, size_t bytes) {
    char path[1024];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f) return 1;
    size_t n = fwrite(p, 1, bytes, f);
    fclose(f);
    return n != bytes;
}

int main(int argc, char** argv) {
    if (argc != 7) {
        printf("usage: usp_step dir S H D U R\n");
        return 2;
    }
    const char* dir = argv[1];
    const int S = atoi(argv[2]), H = atoi(argv[3]), D = atoi(argv[4]), U = atoi(argv[5]), R = atoi(argv[6]);
    const int B = 1;
    dit_sp_layout L;
    CK(dit_sp_layout_init(B, S, H, D, U, R, &L));

    const size_t plane = (size_t)B * S * H * D * 2;          /* bf16 */
    const size_t N = (size_t)S * H * D;                      /* CFG elements per branch */
    void* hq = read_file(dir, "q.bin", plane);
    void* hk = read_file(dir, "k.bin", plane);
    void* hv = read_file(dir, "v.bin", plane);
    void* hp = read_file(dir, "pred.bin", 2 * N * 2);
    if (!hq || !hk || !hv || !hp) {
        printf("FAIL reading inputs\n");
        return 1;
    }

    /* element counts of the buffers (all caller-owned) */
    const size_t wire3 = (size_t)3 * B * L.S_pad * L.Hp * D, wire1 = wire3 / 3;
    const size_t head = (size_t)R * B * L.S_cap * L.Hp * D;
    const size_t parts = (size_t)R * head;                   /* [R][R][B][S_cap][Hp][D] */
    const size_t lse = (size_t)R * R * B * L.Hp * L.S_cap;   /* [R][R][B][Hp][S_cap] */
    void *q, *k, *v, *send, *recv, *qh, *kh, *vh, *part, *oh, *send_o, *recv_o, *out, *pred, *cfg;
    float* lse_p;
    int* status;
    CU(cudaMalloc(&q, plane));
    CU(cudaMalloc(&k, plane));
    CU(cudaMalloc(&v, plane));
    CU(cudaMalloc(&send, wire3 * 2));
    CU(cudaMalloc(&recv, wire3 * 2));
    CU(cudaMalloc(&qh, head * 2));
    CU(cudaMalloc(&kh, head * 2));
    CU(cudaMalloc(&vh, head * 2));
    CU(cudaMalloc(&part, parts * 4));
    CU(cudaMalloc((void**)&lse_p, lse * 4));
    CU(cudaMalloc(&oh, head * 2));
    CU(cudaMalloc(&send_o, wire1 * 2));
    CU(cudaMalloc(&recv_o, wire1 * 2));
    CU(cudaMalloc(&out, plane));
    CU(cudaMalloc(&pred, 2 * N * 2));
    CU(cudaMalloc(&cfg, N * 2));
    CU(cudaMalloc((void**)&status, sizeof(int)));
    CU(cudaMemset(status, 0, sizeof(int)));
    CU(cudaMemcpy(q, hq, plane, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(k, hk, plane, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(v, hv, plane, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(pred, hp, 2 * N * 2, cudaMemcpyHostToDevice));

    /* seq -> head: pack, exchange, unpack with V as f16 */
    const void* src3[3] = {q, k, v};
    void* heads[3] = {qh, kh, vh};
    const dit_dtype head_dt[3] = {DIT_BF16, DIT_BF16, DIT_F16};
    CK(dit_ulysses_pack(&L, DIT_SEQ_TO_HEAD, 3, src3, DIT_BF16, send, DIT_BF16, NULL));
    CK(dit_a2a_sim(&L, DIT_SEQ_TO_HEAD, 3, send, recv, DIT_BF16, NULL));
    CK(dit_ulysses_unpack(&L, DIT_SEQ_TO_HEAD, 3, recv, DIT_BF16, heads, head_dt, status, NULL));

    /* every (ring block r, ring block j) partial: fp32 O, natural-log lse */
    const int64_t sd = D, ss = (int64_t)L.Hp * D, sb = (int64_t)L.S_cap * ss, sr = (int64_t)B * sb;
    dit_view qv = {qh, sr, 0, sb, ss, sd}, kv = {kh, 0, sr, sb, ss, sd}, vv = {vh, 0, sr, sb, ss, sd};
    dit_view pv = {part, (int64_t)R * sr, sr, sb, ss, sd};
    const int64_t ls = L.S_cap, lb = (int64_t)L.Hp * ls, lkv = (int64_t)B * lb;
    dit_lse_view lv = {lse_p, (int64_t)R * lkv, lkv, lb, ls};
    const float scale = 1.0f / sqrtf((float)D);
    CK(dit_attn_partial(B, H, D, scale, R, L.ring_real, R, L.ring_real, qv, DIT_BF16, kv, vv, DIT_F16, pv, DIT_F32,
                        lv, status, NULL));
    /* the ring merge into the head layout (bf16) */
    dit_view ov = {oh, sr, 0, sb, ss, sd};
    dit_lse_view none = {NULL, 0, 0, 0, 0};
    CK(dit_attn_merge_lse(B, H, D, R, L.ring_real, R, pv, DIT_F32, lv, ov, DIT_BF16, none, NULL));

    /* head -> seq: pack, exchange, unpack */
    const void* src1[1] = {oh};
    void* dst1[1] = {out};
    const dit_dtype out_dt[1] = {DIT_BF16};
    CK(dit_ulysses_pack(&L, DIT_HEAD_TO_SEQ, 1, src1, DIT_BF16, send_o, DIT_BF16, NULL));
    CK(dit_a2a_sim(&L, DIT_HEAD_TO_SEQ, 1, send_o, recv_o, DIT_BF16, NULL));
    CK(dit_ulysses_unpack(&L, DIT_HEAD_TO_SEQ, 1, recv_o, DIT_BF16, dst1, out_dt, NULL, NULL));

    /* classifier-free guidance, g = 3.5 */
    CK(dit_cfg_combine(pred, DIT_BF16, (int64_t)N, 3.5f, cfg, DIT_BF16, NULL));
    CU(cudaDeviceSynchronize());

    int st = -1;
    CU(cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost));
    void* ho = malloc(plane);
    void* hc = malloc(N * 2);
    CU(cudaMemcpy(ho, out, plane, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(hc, cfg, N * 2, cudaMemcpyDeviceToHost));
    if (write_file(dir, "out.bin", ho, plane) || write_file(dir, "cfg.bin", hc, N * 2)) {
        printf("FAIL writing outputs\n");
        return 1;
    }
    printf("ok status=%d\n", st);
    return 0;
}
