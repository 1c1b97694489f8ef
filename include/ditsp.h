/*
 * ditsp.h -- C ABI of the GB300 sequence-parallel DiT attention hot path.
 *
 * One shared library, libditsp.so, exposes the steps of sequence-parallel
 * attention for diffusion transformers as plain C calls on device pointers:
 *
 *   dit_sp_layout_init / dit_sp_a2a_counts   rank partition bookkeeping
 *   dit_ulysses_pack / dit_a2a_sim / dit_ulysses_unpack
 *                                            the Ulysses all-to-all, both ways
 *   dit_ulysses_pack_joint / dit_ulysses_unpack_joint
 *                                            the same for paired text/image
 *                                            streams (joint sequence)
 *   dit_ulysses_unpack_rope                  receive preparation with RoPE
 *   dit_ulysses_seq_to_head / dit_ulysses_head_to_seq
 *                                            pack, exchange and unpack in one
 *                                            pass (ranks sharing one memory)
 *   dit_sp_signal / dit_a2a_sim_checked      the exchange with arrival counters
 *                                            and a bounded wait
 *   dit_attn_partial                         attention of query blocks against
 *                                            key/value chunks, with log-sum-exp
 *   dit_attn_merge_lse                       exact merge of the partials
 *   dit_attn_ring                            the partials of every key block
 *                                            folded in as the CTA walks them
 *   dit_attn_ring_rows                       the same, each query block's
 *                                            output placed at its own row
 *   dit_attn_ring_merge_static               partials + merge with the
 *                                            partials in the library's own
 *                                            fixed device array
 *   dit_attention                            single-shot attention
 *   dit_cfg_combine                          classifier-free guidance combine
 *
 * The "ranks" of Ulysses (degree U) and ring (degree R) parallelism are
 * partitions of buffers in one GPU's memory.  Virtual rank id = r*U + u:
 * ring blocks outer, Ulysses ranks inner, so ranks in id order cover the
 * sequence in order (SGLang Diffusion "Parallelism Overview": Ulysses groups
 * on contiguous ranks, ring groups strided).
 *
 * Conventions shared by every call
 *  - Ownership: the caller allocates and owns every buffer.  The library
 *    allocates no device or host memory in any call.  Its one piece of
 *    device memory is the fixed scratch array of dit_attn_ring_merge_static,
 *    part of its device code (DIT_RING_STATIC_SCRATCH_BYTES per device).
 *  - Asynchrony: every call that takes `stream` (a cudaStream_t passed as
 *    void*, NULL = legacy default stream) validates its arguments on the
 *    host, enqueues its kernels on that stream and returns without waiting.
 *  - Errors: argument problems are reported synchronously as
 *    DIT_ERR_INVALID_ARG / DIT_ERR_UNSUPPORTED before anything is launched;
 *    a failed launch returns DIT_ERR_CUDA.  dit_last_error() then holds a
 *    one-line description (per calling thread).  Conditions found on the
 *    device (a bounded wait that ran out, a value out of a target type's
 *    range) are written to a caller-supplied device int `d_status`, or to
 *    the library's own device word when d_status is NULL; read the latter
 *    with dit_device_status().  Nothing traps and nothing crosses the ABI
 *    as an exception.
 *  - Threads: calls hold no global mutable host state except the
 *    thread-local error string and a once-initialised driver entry point.
 *  - Element types: DIT_F32, DIT_BF16, DIT_F16.  Narrowing conversions round
 *    to nearest even; widening is exact.
 *  - Pointers passed to kernels must be 16-byte aligned and every tensor's
 *    innermost (head-dim) extent in bytes a multiple of 16.
 *  - Empty work: a call with nothing to read or write (a layout with S = 0,
 *    attention or a merge with no query rows, a CFG combine with N = 0)
 *    checks its other arguments, launches nothing and returns DIT_OK; its
 *    buffer pointers may then be NULL, as an allocator gives for zero bytes.
 *    Attention whose every key block is empty writes O = 0 and lse = -inf
 *    and may take NULL K and V.
 */
#ifndef DITSP_H
#define DITSP_H

#include <stdint.h>

#if defined(__GNUC__)
#define DIT_API __attribute__((visibility("default")))
#else
#define DIT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DIT_OK = 0,
    DIT_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment */
    DIT_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head dim) */
    DIT_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    DIT_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out */
    DIT_ERR_RANGE = 5          /* a value overflowed the target type */
} dit_status;

/* DIT_E4M3 is a wire type only (dit_ulysses_pack / dit_a2a_sim /
 * dit_ulysses_unpack and their variants): one record per (token, head) of D
 * e4m3 codes, the head's float32 scale and 12 zero bytes (D + 16 bytes);
 * see dit_ulysses_pack. */
typedef enum { DIT_F32 = 0, DIT_BF16 = 1, DIT_F16 = 2, DIT_E4M3 = 3 } dit_dtype;

/* Direction of a Ulysses exchange (edge-dit.cpp "Parallel execution",
 * SPAllToAll4DLayout: kSeqToHead / kHeadToSeq). */
typedef enum { DIT_SEQ_TO_HEAD = 0, DIT_HEAD_TO_SEQ = 1 } dit_a2a_dir;

#define DIT_MAX_U 64
#define DIT_MAX_R 8
#define DIT_MAX_RANKS 64
/* bytes of the fixed scratch array of dit_attn_ring_merge_static */
#define DIT_RING_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * Rank partition of one sequence-parallel attention (edge-dit.cpp
 * "Parallel execution", SPSequenceSplit and SPAllToAll4DLayout; cache-dit
 * "Context Parallelism", UAA and Any Head Num).
 *
 * The S_pad rows of the sequence are split over R ring blocks and each ring
 * block over U Ulysses ranks with the balanced rule: of n parts the first
 * S_pad mod n get one extra row (lengths differ by at most one).  Rows at or
 * past S are sequence padding (S_pad = S unless DIT_LAYOUT_PAD_LCM64).
 * Ulysses rank v owns head_len[v] head slots starting at head_off[v]; head
 * slots at or past H are zero.  By default heads are padded from H to
 * Hp = ceil(H/U)*U and every group has Hl = Hp/U slots.
 *
 * Layout flags (dit_sp_layout_init_ex):
 *   DIT_LAYOUT_NOPAD_HEADS  no head padding (cache-dit "Context
 *     Parallelism", the padding-free variant of Any Head Num): head_len is
 *     the balanced split of H (the first H mod U groups one more), Hp = H,
 *     Hl = the largest group.
 *   DIT_LAYOUT_PAD_LCM64    sequence padding (xLLM "DiT Architecture and
 *     Capability Matrix": with SP the total length is padded to a multiple
 *     of lcm(SP, 64) before partitioning): S_pad = S rounded up to a
 *     multiple of lcm(U*R, 64).  Padding rows travel as zeros, are excluded
 *     from attention by passing each ring block's real row count, and are
 *     dropped by the head-to-seq unpack.
 */
#define DIT_LAYOUT_NOPAD_HEADS 1
#define DIT_LAYOUT_PAD_LCM64 2

typedef struct {
    int B, S, H, D, U, R;
    int Hp, Hl;                       /* head slots in total / in the largest group */
    int S_cap;                        /* max ring-block length */
    int ring_len[DIT_MAX_R];          /* rows of ring block r */
    int ring_off[DIT_MAX_R];          /* first global row of ring block r */
    int rank_len[DIT_MAX_RANKS];      /* rows of virtual rank r*U+u */
    int rank_off[DIT_MAX_RANKS];      /* first global row of that rank */
    int S_pad;                        /* rows split over the ranks (>= S) */
    int flags;                        /* DIT_LAYOUT_* */
    int head_len[DIT_MAX_U];          /* head slots of Ulysses rank v */
    int head_off[DIT_MAX_U];          /* first head slot of Ulysses rank v */
    int ring_real[DIT_MAX_R];         /* rows of ring block r that are real
                                         (< S): its attention query and key
                                         counts */
} dit_sp_layout;

/*
 * A strided view of a [blocks][B][rows][heads][D] tensor; d is contiguous.
 * Strides are in elements.  stride_q steps between query (ring) blocks,
 * stride_kv between key/value blocks (for partial outputs: the partial of
 * query block r against key/value block j is at r*stride_q + j*stride_kv).
 * A stride that a call does not use is ignored.
 */
typedef struct {
    void* ptr;
    int64_t stride_q, stride_kv, stride_b, stride_s, stride_h;
} dit_view;

/* A strided view of float32 log-sum-exp rows [blocks][B][heads][rows];
 * rows are contiguous. */
typedef struct {
    float* ptr;
    int64_t stride_q, stride_kv, stride_b, stride_h;
} dit_lse_view;

DIT_API const char* dit_status_string(dit_status s);

/* One-line description of the last error returned on this thread. */
DIT_API const char* dit_last_error(void);

/* Reads (and if reset != 0 clears) the library's own device status word,
 * used by calls whose d_status is NULL.  Synchronises the device. */
DIT_API dit_status dit_device_status(int* out_code, int reset);

/*
 * dit_sp_layout_init: fill *out for a [B, S, H, D] attention split over
 * U Ulysses ranks inside R ring blocks.  Host only, no device work.
 * Requires B,H,D >= 1, S >= 0, 1 <= U <= DIT_MAX_U, 1 <= R <= DIT_MAX_R,
 * U*R <= DIT_MAX_RANKS, and every size product within int64.
 */
DIT_API dit_status dit_sp_layout_init(int B, int S, int H, int D, int U, int R,
                              dit_sp_layout* out);

/* dit_sp_layout_init_ex: as dit_sp_layout_init with DIT_LAYOUT_* flags
 * (0 gives dit_sp_layout_init); other bits are DIT_ERR_INVALID_ARG. */
DIT_API dit_status dit_sp_layout_init_ex(int B, int S, int H, int D, int U, int R, int flags,
                                 dit_sp_layout* out);

/*
 * dit_sp_a2a_counts: the alltoallv argument set of virtual rank `rank` for
 * one exchange carrying `nplanes` planes (3 = packed Q,K,V; 1 = O), in
 * elements, indexed by the peer's Ulysses index within the rank's ring
 * group.  Send blocks are peer-major; the block rank u sends rank v is
 * [nplanes][B][rows][heads][D] with rows = rank_len of u (seq-to-head) or
 * of v (head-to-seq) and heads = head_len of v (seq-to-head) or of u
 * (head-to-seq).  Each output array has room for U entries.  Host only.
 */
DIT_API dit_status dit_sp_a2a_counts(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                             int rank, int64_t* send_counts, int64_t* send_displs,
                             int64_t* recv_counts, int64_t* recv_displs);

/*
 * Buffer shapes used by the Ulysses calls (all dense, row-major):
 *   seq layout   [B][S][H][D]              rank (r,u) owns rows
 *                                          [rank_off, rank_off + rank_len)
 *                                          (the real ones: rows < S)
 *   head layout  [R][B][S_cap][Hp][D]      rank (r,v) owns ring block r,
 *                                          rows [0, ring_len[r]), head
 *                                          slots [head_off[v], head_off[v]
 *                                          + head_len[v]); rows past
 *                                          ring_len[r] are never touched
 *   wire         all ranks' send (or receive) buffers end to end in rank-id
 *                order; total nplanes*B*S_pad*Hp*D elements
 * Sequence-padding rows (>= S) are zero on the wire in both directions and
 * zero in the head layout after the seq-to-head unpack.
 *
 * dit_ulysses_pack (edge-dit.cpp "Parallel execution": packed QKV send path
 * and head-to-sequence path).
 *   DIT_SEQ_TO_HEAD: src[p] (p < nplanes) are seq-layout planes; every rank
 *     writes, for each destination v in order, its rows of head group v of
 *     every plane; heads >= H are written as zero.
 *   DIT_HEAD_TO_SEQ: src[0] is a head-layout tensor (nplanes must be 1);
 *     rank (r,v) writes, for each destination u, u's rows of its heads;
 *     heads >= H are written as zero.
 *   Values are converted src_dt -> wire_dt.
 *
 * dit_a2a_sim: the exchange itself: every rank's receive buffer is the
 *   concatenation, over source ranks in order, of the blocks they addressed
 *   to it.  A permutation copy in one memory; no arithmetic.
 *
 * dit_ulysses_unpack:
 *   DIT_SEQ_TO_HEAD: dst[p] are head-layout planes, converted wire_dt ->
 *     dst_dt[p] (e.g. Q,K bf16 and V f16).  If d_range_flag is not NULL,
 *     a value that overflows dst_dt[p] sets *d_range_flag = DIT_ERR_RANGE
 *     (the converted value is the rounded infinity).
 *   DIT_HEAD_TO_SEQ: dst[0] is a seq-layout tensor [B][S][H][D] in dst_dt[0];
 *     padded heads are dropped.
 *
 * The three calls require D to be a multiple of 8 (so that a head row is a
 * multiple of 16 bytes in every type; else DIT_ERR_UNSUPPORTED) and 16-byte
 * aligned pointers.  send/recv must not
 * overlap any other buffer of the same call.
 *
 * wire_dt = DIT_E4M3 (cache-dit "Context Parallelism", Async FP8 Ulysses
 * Attention: Q, V and O cross the all-to-all in float8, K stays 16-bit):
 * every (token, head) travels as a record of D + 16 bytes, the send and
 * receive buffers hold nplanes*B*S*Hp records in the wire order above.  The
 * pack computes, in IEEE float32 with round to nearest even,
 *   amax = max |x_d|,  s = amax / 448,  r = 1 / s (0 when s = 0),
 *   code_d = e4m3(x_d * r) with saturation to +-448,
 * and writes the D codes, s (float32) and 12 zero bytes; padded heads are
 * zero records.  The unpack writes code_d * s (float32) rounded to dst_dt.
 * dit_a2a_sim moves records unchanged.  D must be 16, 32, 64, 128 or 256
 * (else DIT_ERR_UNSUPPORTED); inputs must be finite (a head holding an
 * infinity or NaN gets an unspecified record).  Keep K on a 16-bit wire.
 */
DIT_API dit_status dit_ulysses_pack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                            const void* const* src, dit_dtype src_dt,
                            void* send, dit_dtype wire_dt, void* stream);

DIT_API dit_status dit_a2a_sim(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                       const void* send, void* recv, dit_dtype wire_dt, void* stream);

/*
 * Checked exchange (SGLang Diffusion "Parallelism Overview", The Ulysses
 * transport: senders publish GPU-side sequence counters instead of a
 * rendezvous, and a timeout backstop makes the request fail rather than
 * return incomplete data).
 *
 * dit_sp_signal: every virtual rank i with rank_mask[i] != 0 (all ranks if
 *   rank_mask is NULL; host array of U*R bytes) publishes `epoch` on its
 *   arrival counter d_arrival[i] (device, U*R unsigned ints, caller-owned).
 *   Stream-ordered: issue it after the pack that fills the send buffers.
 * dit_a2a_sim_checked: as dit_a2a_sim, but each run is copied only once its
 *   sender's counter has reached `epoch` (unsigned sequence comparison).  A
 *   counter that does not get there within timeout_ns (0 < t <= 10 s) sets
 *   *d_status = DIT_ERR_TIMEOUT (the library's word if d_status is NULL) and
 *   the rest of the exchange is abandoned: runs whose senders timed out are
 *   not written, and the receive buffer must be treated as invalid.  The
 *   kernel always returns; the device stays usable.  The status word must
 *   not hold DIT_ERR_TIMEOUT when the call starts: the kernel reads it to
 *   abandon the exchange at once, so a stale value from an earlier call makes
 *   every wait give up immediately (clear it, e.g. dit_device_status with
 *   reset = 1 for the library's word).  The signalling side publishes with
 *   a release (a fence before the counter store) and the waiting side
 *   fences after observing the counter, so a sender that is not stream
 *   ordered with the exchange is read in full.
 */
DIT_API dit_status dit_sp_signal(const dit_sp_layout* L, unsigned* d_arrival, const unsigned char* rank_mask,
                                 unsigned epoch, void* stream);

DIT_API dit_status dit_a2a_sim_checked(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                                       const void* send, void* recv, dit_dtype wire_dt,
                                       const unsigned* d_arrival, unsigned epoch, int64_t timeout_ns,
                                       int* d_status, void* stream);

DIT_API dit_status dit_ulysses_unpack(const dit_sp_layout* L, dit_a2a_dir dir, int nplanes,
                              const void* recv, dit_dtype wire_dt,
                              void* const* dst, const dit_dtype* dst_dt,
                              int* d_range_flag, void* stream);

/*
 * Paired text and image streams (edge-dit.cpp "Parallel execution": the
 * packed QKV path has a variant for the paired streams of FLUX double-stream
 * blocks, decoded and assembled into the joint attention sequence).  The
 * joint sequence is the S_txt text tokens followed by the S - S_txt image
 * tokens; the layout L splits the joint sequence as usual, so a rank's rows
 * may come from either stream or both.
 *
 * dit_ulysses_pack_joint: as dit_ulysses_pack(DIT_SEQ_TO_HEAD), with plane p
 *   read from txt[p] ([B][S_txt][H][D]) for joint rows t < S_txt and from
 *   img[p] ([B][S - S_txt][H][D]) at row t - S_txt for the others.  0 <= S_txt
 *   <= S; txt (img) may be NULL when S_txt == 0 (S_txt == S).  The send
 *   buffer is bit-identical to dit_ulysses_pack of the concatenated planes.
 * dit_ulysses_unpack_joint: as dit_ulysses_unpack(DIT_HEAD_TO_SEQ), writing
 *   joint rows t < S_txt to out_txt [B][S_txt][H][D] and the others to
 *   out_img [B][S - S_txt][H][D] at row t - S_txt, in out_dt.
 * Errors and alignment as for dit_ulysses_pack / dit_ulysses_unpack.
 */
DIT_API dit_status dit_ulysses_pack_joint(const dit_sp_layout* L, int nplanes, const void* const* txt,
                                          const void* const* img, int S_txt, dit_dtype src_dt, void* send,
                                          dit_dtype wire_dt, void* stream);

DIT_API dit_status dit_ulysses_unpack_joint(const dit_sp_layout* L, const void* recv, dit_dtype wire_dt,
                                            void* out_txt, void* out_img, int S_txt, dit_dtype out_dt,
                                            void* stream);

/*
 * dit_ulysses_unpack_rope: the receive preparation (edge-dit.cpp "Parallel
 * execution": one pass decodes the rank-major receive buffer, extracts the
 * Q/K/V planes, writes the head-sharded layout and applies RoPE to Q and K,
 * with V in its attention layout).  As dit_ulysses_unpack(DIT_SEQ_TO_HEAD),
 * except that every plane p with bit p of rope_planes set is rotated while
 * it is written: for the token at joint-sequence position t and each pair
 * i < D/2 of every head,
 *   y[2i]   = x[2i] * cos_tab[t*D/2 + i] - x[2i+1] * sin_tab[t*D/2 + i]
 *   y[2i+1] = x[2i] * sin_tab[t*D/2 + i] + x[2i+1] * cos_tab[t*D/2 + i]
 * with x the received value in fp32, computed in fp32 (one rounded product
 * and one fused multiply-add per output) and rounded to dst_dt[p].
 *   cos_tab, sin_tab  device, float32 [S][D/2] row-major, 16-byte aligned,
 *                     caller-owned (the model's angles: the pages give none).
 *   rope_planes       bit mask over the nplanes planes (0x3 = Q and K);
 *                     0 gives dit_ulysses_unpack exactly.
 * Padded heads are not rotated and stay +0.  d_range_flag as for
 * dit_ulysses_unpack (a 16-bit
 * destination value that becomes infinite sets it).  On a 16- or 32-bit wire
 * the rotation needs D <= 384 (else DIT_ERR_UNSUPPORTED); the e4m3 wire takes
 * its own D set.
 */
DIT_API dit_status dit_ulysses_unpack_rope(const dit_sp_layout* L, int nplanes, const void* recv,
                                           dit_dtype wire_dt, void* const* dst, const dit_dtype* dst_dt,
                                           const float* cos_tab, const float* sin_tab, unsigned rope_planes,
                                           int* d_range_flag, void* stream);

/*
 * One-pass permutation (edge-dit.cpp "Parallel execution": packed QKV send
 * path, receive preparation and head-to-sequence path; SGLang Diffusion
 * "Parallelism Overview", The Ulysses transport).  When every virtual rank
 * lives in one memory, rank v's receive block from u is rank u's send block
 * to v, so the exchange may alias the two (recv[v][u] == send[u][v]) and
 * pack, exchange and unpack compose into one pass that reads each element
 * once and writes it once, with no send or receive buffer.  The results are
 * bit-identical to the three calls with the wire in the source type.
 *
 * Sequence-side tensors come in one piece or as a pair split at row
 * `split` (the paired text/image streams of a double-stream block): rows
 * t < split in src[p] ([B][split][H][D]) and rows t >= split in src2[p]
 * ([B][S - split][H][D]) at row t - split.  split = 0 (or S): src[p] holds
 * all S rows ([B][S][H][D]) and src2 is not read (may be NULL).
 *
 * dit_ulysses_seq_to_head: head-layout planes dst[p] ([R][B][S_cap][Hp][D],
 *   dst_dt[p]) from the sequence-layout planes: row i of ring block r, batch
 *   b = sequence row ring_off[r] + i, its H heads converted src_dt ->
 *   dst_dt[p] (one rounding) and Hp - H zero heads; sequence-padding rows
 *   are zero; rows past ring_len[r] are not touched.  Planes with bit p of
 *   rope_planes set are rotated as by dit_ulysses_unpack_rope (cos_tab,
 *   sin_tab float32 [S][D/2], 16-byte aligned; NULL when rope_planes = 0;
 *   D <= 384 when rope_planes != 0, else DIT_ERR_UNSUPPORTED).
 *   d_range_flag as for dit_ulysses_unpack.  Equal to dit_ulysses_pack (or
 *   _pack_joint) + dit_a2a_sim + dit_ulysses_unpack (or _unpack_rope) with
 *   wire_dt = src_dt.
 * dit_ulysses_head_to_seq: the sequence-layout output (dst / dst2 split as
 *   above, [B][S][H][D] in dst_dt) from a head-layout tensor src (src_dt):
 *   row t < S = the first H heads of head-layout row (r, b, t - ring_off[r]).
 *   Equal to dit_ulysses_pack + dit_a2a_sim + dit_ulysses_unpack (or
 *   _unpack_joint) with wire_dt = src_dt.
 * Both: D a multiple of 8, pointers 16-byte aligned, destination types of
 * one size per call; a layout with S = 0 moves nothing.  Source and
 * destination must not overlap.
 */
DIT_API dit_status dit_ulysses_seq_to_head(const dit_sp_layout* L, int nplanes, const void* const* src,
                                           const void* const* src2, int split, dit_dtype src_dt,
                                           void* const* dst, const dit_dtype* dst_dt, const float* cos_tab,
                                           const float* sin_tab, unsigned rope_planes, int* d_range_flag,
                                           void* stream);

DIT_API dit_status dit_ulysses_head_to_seq(const dit_sp_layout* L, const void* src, dit_dtype src_dt, void* dst,
                                           void* dst2, int split, dit_dtype dst_dt, void* stream);

/*
 * dit_attn_partial: for every query block r < n_q and key/value block
 * j < n_kv, the attention of Q_r against the first kv_len[j] keys of
 * (K_j, V_j) (SGLang Diffusion "Parallelism Overview", Constraints: the
 * ring's per-hop merge needs each call's softmax log-sum-exp; diffusers
 * "Distributed inference", Ring Anything: padded K/V trimmed to the real
 * length).  For each batch b, head h < H and row i < q_len[r]:
 *   s_t   = scale * <q_i, k_t>              for keys t < kv_len[j]
 *   lse_i = ln sum_t exp(s_t)
 *   o_i   = sum_t exp(s_t - lse_i) * v_t    (normalised by this chunk only)
 * Keys at or past kv_len[j] are excluded from the softmax, whatever their
 * contents.  A chunk with kv_len[j] == 0 gives o = 0 and lse = -inf.
 * scale must be positive and finite (1/sqrt(D) in the pages' attention).
 *
 *   q        rows of block r at q.ptr + r*q.stride_q, [B][q_len[r]][H][D]
 *   k, v     rows of block j at ptr + j*stride_kv,    [B][kv_len[j]][H][D]
 *   o        partial (r, j) at o.ptr + r*o.stride_q + j*o.stride_kv
 *   lse      partial (r, j) row i of (b, h) at
 *            r*stride_q + j*stride_kv + b*stride_b + h*stride_h + i;
 *            lse.ptr may be NULL (not written)
 *   q_len, kv_len: host arrays; n_q, n_kv <= DIT_MAX_R.
 *
 * Supported: (qk_dt, v_dt) = (F32, F32) with o_dt F32 and D in {16, 32,
 * 64, 128} (fp32 CUDA-core path); or qk_dt in {BF16, F16}, v_dt in {BF16,
 * F16}, D in {64, 128}, o_dt in {F32, BF16, F16} (tensor-core path: Q K^T
 * in qk_dt with fp32 accumulation; P rounded to v_dt for P V with fp32
 * accumulation).  Strides and pointers must be 16-byte aligned.  Each o row
 * is a convex combination of V rows, so o_dt = F16 cannot overflow when
 * v_dt is F16.
 * Head dims other than these return DIT_ERR_UNSUPPORTED.  The output view
 * must give every result its own address: a zero o stride on a dimension
 * with more than one index (stride_h with H > 1, stride_s with a block of
 * more than one row, stride_b with B > 1, stride_q / stride_kv with more
 * than one block) returns DIT_ERR_INVALID_ARG.
 */
DIT_API dit_status dit_attn_partial(int B, int H, int D, float scale,
                            int n_q, const int* q_len, int n_kv, const int* kv_len,
                            dit_view q, dit_dtype qk_dt, dit_view k, dit_view v,
                            dit_dtype v_dt, dit_view o, dit_dtype o_dt,
                            dit_lse_view lse, int* d_status, void* stream);

/*
 * dit_attn_ring: ring attention of every query block r < n_q against all its
 * key/value blocks j < n_kv, folded into one exact result per query block
 * (SGLang Diffusion "Parallelism Overview", What happens to the shapes and
 * Constraints: Q stays in place while the K/V chunks of the ring group visit,
 * and each hop is folded in with the online softmax).  For each batch b,
 * head h and row i < q_len[r], over every key t < kv_len[j] of every block j:
 *   o_i   = sum_t softmax_t(scale * <q_i, k_t>) v_t
 *   lse_i = ln sum_t exp(scale * <q_i, k_t>)
 * which equals dit_attn_partial followed by dit_attn_merge_lse up to
 * rounding.  The kernel walks the blocks in order with one running row max,
 * sum and O accumulator (in TMEM on the tensor-core path), so no partial is
 * written.  Blocks with kv_len[j] == 0 are skipped; a query block whose every
 * key block is empty gets o = 0, lse = -inf.
 *   q, k, v   as for dit_attn_partial
 *   o         query block r at o.ptr + r*o.stride_q, [B][q_len[r]][H][D]
 *             (o.stride_kv is ignored)
 *   lse       row i of (r, b, h) at r*stride_q + b*stride_b + h*stride_h + i
 *             (stride_kv ignored); lse.ptr may be NULL
 * Types, head dims, alignment and the output-aliasing rule as for
 * dit_attn_partial.
 */
DIT_API dit_status dit_attn_ring(int B, int H, int D, float scale, int n_q, const int* q_len, int n_kv,
                                 const int* kv_len, dit_view q, dit_dtype qk_dt, dit_view k, dit_view v,
                                 dit_dtype v_dt, dit_view o, dit_dtype o_dt, dit_lse_view lse, int* d_status,
                                 void* stream);

/*
 * dit_attn_ring_rows: dit_attn_ring with each query block's output moved
 * o_row0[r] rows further into o:
 *   o         query block r at o.ptr + r*o.stride_q + o_row0[r]*o.stride_s,
 *             [B][q_len[r]][H][D]
 * When every rank lives in one memory, the head-to-sequence exchange of the
 * output (edge-dit.cpp "Parallel execution", head-to-sequence path) only
 * moves ring block r's rows to rows ring_off[r] + i of the sequence layout
 * and drops the padded heads; with o.stride_q = 0, o_row0[r] = ring_off[r]
 * and the sequence layout's strides, the attention writes each result at
 * that place and no layout pass follows.  The lse rows are not moved.
 * o_row0 is a host array of n_q entries >= 0.  With o.stride_q == 0 the
 * blocks' output rows [o_row0[r], o_row0[r] + q_len[r]) must not overlap
 * (DIT_ERR_INVALID_ARG otherwise).  Everything else as for dit_attn_ring.
 */
DIT_API dit_status dit_attn_ring_rows(int B, int H, int D, float scale, int n_q, const int* q_len,
                                      const int* o_row0, int n_kv, const int* kv_len, dit_view q,
                                      dit_dtype qk_dt, dit_view k, dit_view v, dit_dtype v_dt, dit_view o,
                                      dit_dtype o_dt, dit_lse_view lse, int* d_status, void* stream);

/*
 * dit_attn_varlen: attention of packed variable-length sequences (SGLang
 * Diffusion "Parallelism Overview", the generic varlen path with several
 * packed segments per row; xLLM "DiT Architecture and Capability Matrix",
 * packed TND data with live/padding boundaries).  Sequence s < nseq has
 * query rows [cu_q[s], cu_q[s+1]) and key rows [cu_k[s], cu_k[s+1]) and
 * attends only to its own keys:
 *   o_i = sum_t softmax_t(scale * <q_i, k_t>) v_t,  lse_i = ln sum_t exp(...)
 * over its keys t; a sequence with no keys gives o = 0, lse = -inf.  Rows of
 * q outside every sequence are not written.
 *   q, o     packed rows [Tq][H][D]: row t at ptr + t*stride_s + h*stride_h
 *   k, v     packed rows [Tk][H][D]
 *   lse      [H][Tq] at lse.ptr + h*stride_h + t (may be NULL)
 *   cu_q, cu_k  host arrays of nseq + 1 non-decreasing row offsets.
 * Block and batch strides of the views are ignored.  Types, head dims and
 * alignment as for dit_attn_partial; the library issues one launch per
 * DIT_MAX_R sequences.
 */
DIT_API dit_status dit_attn_varlen(int H, int D, float scale, int nseq, const int* cu_q, const int* cu_k,
                                   dit_view q, dit_dtype qk_dt, dit_view k, dit_view v, dit_dtype v_dt,
                                   dit_view o, dit_dtype o_dt, dit_lse_view lse, int* d_status, void* stream);

/*
 * dit_attn_merge_lse: fold n_parts partials of each query block into the
 * exact result (SGLang Diffusion "Parallelism Overview", What happens to the
 * shapes and Constraints: online-softmax merge over ranks holding the same
 * heads over different rows).  For each (r, b, h, i):
 *   M   = max_j lse_j,   lse = M + ln sum_j exp(lse_j - M)
 *   out = sum_j exp(lse_j - lse) * O_j          (j ascending, fp32)
 * Rows whose every partial is empty (lse_j = -inf) give out = 0, lse = -inf.
 *   parts:  partial j of block r at parts.ptr + r*stride_q + j*stride_kv
 *   lse_parts: same indexing as dit_attn_partial's lse
 *   out:    block r at out.ptr + r*out.stride_q; lse_out may have ptr NULL
 * parts_dt in {F32, BF16, F16}; out_dt in {F32, BF16, F16}; D % 8 == 0.
 */
DIT_API dit_status dit_attn_merge_lse(int B, int H, int D, int n_q, const int* q_len,
                              int n_parts, dit_view parts, dit_dtype parts_dt,
                              dit_lse_view lse_parts, dit_view out, dit_dtype out_dt,
                              dit_lse_view lse_out, void* stream);

/*
 * dit_attn_ring_merge_static: dit_attn_partial followed by
 * dit_attn_merge_lse, with the partials (fp32) and their log-sum-exp rows
 * held in a fixed device array of the library instead of caller memory.
 * The pages have no counterpart of this call: it exists for callers that
 * cannot allocate device memory, e.g. code running inside an engine or
 * framework whose memory pool owns the whole device (a stray cudaMalloc
 * would fail there or break the pool's accounting), or code on a
 * latency-critical path where cudaMalloc/cudaFree would stall on an
 * implicit device synchronisation.
 *
 * Arguments, types, head dims and results are those of dit_attn_ring (the
 * same o and lse layout: query block r at o.ptr + r*o.stride_q, stride_kv
 * ignored); the result equals the caller-buffer pair dit_attn_partial ->
 * dit_attn_merge_lse on fp32 partials, and dit_attn_ring up to rounding.
 *
 * The scratch array:
 *  - size DIT_RING_STATIC_SCRATCH_BYTES (64 MiB), aligned to 256 bytes;
 *    every device on which the library's code is loaded holds it until the
 *    process exits.  One call needs
 *      P = n_q*n_kv*B*H*max_r(q_len[r])*D*4 bytes of partials, rounded up
 *          to a multiple of 256, plus n_q*n_kv*B*H*max_r(q_len[r])*4 bytes
 *          of log-sum-exp rows;
 *    a call that needs more returns DIT_ERR_INVALID_ARG before touching the
 *    device.
 *  - the first call on a device looks up the array's device address on the
 *    current device (cudaGetSymbolAddress) and caches it for the life of the
 *    process (like the library's status word); make that first call outside
 *    any stream capture, and make no call after a cudaDeviceReset of that
 *    device, whose new context may place the array elsewhere.
 *  - every call on a device shares the one array, and it keeps the last
 *    call's contents.  Nothing in it needs clearing: the partial step writes
 *    every value the merge step reads.  Calls that overlap on the GPU (on
 *    different streams, or from several host threads without ordering)
 *    race on it and give wrong results; order them on one stream.
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine.
 */
DIT_API dit_status dit_attn_ring_merge_static(int B, int H, int D, float scale, int n_q, const int* q_len,
                                              int n_kv, const int* kv_len, dit_view q, dit_dtype qk_dt,
                                              dit_view k, dit_view v, dit_dtype v_dt, dit_view o,
                                              dit_dtype o_dt, dit_lse_view lse, int* d_status, void* stream);

/*
 * dit_attention: single-shot attention O = softmax(scale * Q K^T) V over
 * all Sk keys (edge-dit.cpp "Parallel execution", Ulysses sequence
 * parallelism: exact full-sequence attention per head), with the row
 * log-sum-exp if lse.ptr is not NULL.  Same types and layout rules as
 * dit_attn_partial with one query block and one key/value block.
 */
DIT_API dit_status dit_attention(int B, int H, int D, float scale, int Sq, int Sk,
                         dit_view q, dit_dtype qk_dt, dit_view k, dit_view v,
                         dit_dtype v_dt, dit_view o, dit_dtype o_dt,
                         dit_lse_view lse, int* d_status, void* stream);

/*
 * dit_cfg_combine: p = p_uncond + g * (p_cond - p_uncond), elementwise
 * (edge-dit.cpp "Parallel execution", classifier-free guidance; under CFG
 * parallelism rank 0 holds the unconditional branch).  pred is a dense
 * [2][N] tensor: pred[0] unconditional, pred[1] conditional.  Arithmetic in
 * fp32 as fma(g, p_cond - p_uncond, p_uncond), rounded once to out_dt;
 * g = 0 returns p_uncond and g = 1 returns p_cond exactly.  N >= 0; pointers
 * 16-byte aligned; out must not overlap pred.
 */
DIT_API dit_status dit_cfg_combine(const void* pred, dit_dtype in_dt, int64_t N, float g,
                           void* out, dit_dtype out_dt, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DITSP_H */
