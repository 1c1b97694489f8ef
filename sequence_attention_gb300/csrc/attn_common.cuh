// Argument block shared by the two attention implementations (fp32 CUDA
// cores, bf16/f16 tensor cores) and the ABI entry points that dispatch to them.
#pragma once

#include "common.cuh"

namespace ditsp {

struct AttnArgs {
    int B, H, D, n_q, n_kv;
    int q_len[DIT_MAX_R];
    int kv_len[DIT_MAX_R];
    float scale;
    dit_view q, k, v, o;
    dit_dtype qk_dt, v_dt, o_dt;
    dit_lse_view lse;
    int* status;
    // packed variable-length sequences: block i's rows start at row
    // q_row0[i] / kv_row0[i] of the views (0 otherwise), and with diag set
    // query block i attends key block i only (n_q == n_kv)
    int q_row0[DIT_MAX_R];
    int kv_row0[DIT_MAX_R];
    // query block i's output rows start o_row0[i] rows further into o (after
    // q_row0[i]); the lse rows are not moved (0 unless the caller asks)
    int o_row0[DIT_MAX_R];
    int diag;
    // with fold set, every query block walks all key blocks and folds them
    // into one result with the online softmax (the ring's per-hop merge): o
    // and lse have no key-block dimension (their stride_kv is ignored)
    int fold;
};

dit_status launch_attn_f32(const AttnArgs& a, cudaStream_t st);
dit_status launch_attn_tc(const AttnArgs& a, cudaStream_t st);

}  // namespace ditsp
