/* Ulysses sequence-parallel attention block on one GPU: the C ABI.
 *
 * The method (web pages on Ulysses Sequence Parallelism; cited by title and paragraph):
 *   "Snowflake's Ulysses trick trains transformers on million-token contexts across
 *   GPUs", para 2: the sequence is sharded across P ranks; each rank computes its local
 *   QKV projection; an all-to-all leaves every rank the full sequence for a subset of
 *   the attention heads; since heads are independent each rank runs FlashAttention on
 *   its heads; a second all-to-all restores the sequence sharding.  Para 3: two
 *   all-to-alls per layer, total volume O(hidden x seq_len / P).
 *   "Ulysses Sequence Parallelism: Training with Million-Token Contexts" (the Hugging
 *   Face post): para 3 (attention is quadratic; FlashAttention tiles it and never
 *   materialises the score matrix), para 5 (the second all-to-all reverses the first),
 *   para 7 (heads are partitioned across GPUs), para 8 (the input is split along the
 *   sequence dimension).
 *
 * Here the P ranks are virtual: P slices of one GPU's memory.  The all-to-alls are
 * on-device permutation kernels and there is no inter-GPU collective.
 *
 * Notation: S tokens, P ranks, H query heads, G KV heads, D head_dim, C = (H + 2G) * D.
 * Shards are contiguous (rank r owns tokens [r*S/P, (r+1)*S/P)); rank r's head group is
 * query heads [r*H/P, (r+1)*H/P) and KV heads [r*G/P, (r+1)*G/P); query head h reads KV
 * head h / (H/G).  Attention is causal (key j visible to query i iff j <= i).
 *
 * Tensor layouts (row-major, innermost last; "bf16" = 16-bit brain float storage):
 *   x        [S][hidden]                 bf16   token rows; rank r's shard is rows r*S/P..
 *   w        [C][hidden]                 bf16   projection weight, nn.Linear layout,
 *                                               rows = q heads, then k heads, then v heads
 *   qkv_seq  [P][S/P][H + 2G][D]         bf16   (or fp32 when in_fp32): = [S][C]
 *   q        [P][S][H/P][D]              bf16   rank r2's query heads for all tokens
 *   k, v     [P][S][G/P][D]              bf16
 *   o        [P][S][H/P][D]              bf16
 *   lse      [P][H/P][S]                 fp32   natural-log logsumexp of each score row
 *   o_seq    [P][S/P][H][D]              bf16   = [S][H][D]
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers to caller-owned memory, 16-byte aligned.  The library
 *     never frees or keeps them past the call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and return a uly_status at once.  They never throw or exit.
 *   - On error nothing is launched and ulysses_last_error() describes the problem (a
 *     thread-local string valid until the next call on the same thread).
 *   - Device-side failures (a wait that ran out, an input out of range) are recorded in a
 *     status word held by the plan; ulysses_sync_status() reads and clears it.  The word
 *     is sticky: while it holds an error, every kernel of every later call on the same plan
 *     gives up at its first wait that does not complete at once, so those calls' outputs
 *     are undefined.  After a failure, call ulysses_sync_status() (which clears the word)
 *     before relying on the plan again.
 *   - S = 0 is valid: every call is a no-op that returns ULY_OK.
 */
#ifndef ULYSSES_H_
#define ULYSSES_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum uly_status {
  ULY_OK = 0,
  ULY_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
  ULY_ERR_UNSUPPORTED = 2,  /* valid in principle, not built here (e.g. D not 64/128) */
  ULY_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  ULY_ERR_OOM = 4,          /* the plan could not allocate its own small buffers */
  ULY_ERR_TIMEOUT = 5,      /* a device-side wait ran past its limit (from sync_status) */
  ULY_ERR_RANGE = 6,        /* an input's magnitude lies beyond what the backward's scaled
                               fp16 operands can hold (from sync_status) */
  ULY_ERR_BOUNDS = 7        /* debug build (libulysses_debug.so) only: a kernel computed a
                               global index outside its buffer and skipped the access (from
                               sync_status) */
} uly_status;

/* Plan flags. */
#define ULY_FLAG_INJECT_STALL 0x1u /* test only: in block 0 of ulysses_attn_fwd and
                                      ulysses_attn_bwd the MMA issuer withholds its first
                                      score-ready signal, so the bounded waits run out and
                                      the call reports ULY_ERR_TIMEOUT */

typedef struct uly_config {
  int64_t seq_len;        /* S, tokens over all ranks; S % P == 0 */
  int32_t batch;          /* must be 1 */
  int32_t P;              /* virtual ranks (>= 1) */
  int32_t hidden;         /* width of x and of the rows of w; multiple of 8 */
  int32_t n_q_heads;      /* H; H % P == 0 and H % G == 0 */
  int32_t n_kv_heads;     /* G; G % P == 0 */
  int32_t head_dim;       /* D: 64 or 128 */
  int32_t causal;         /* must be 1 */
  int32_t wait_timeout_ms;/* limit of every device-side wait; 0 means 2000 */
  double softmax_scale;   /* 0 means 1/sqrt(D) */
  double rope_theta;      /* > 0 enables rotate-half RoPE in seq_to_head; 0 disables */
  uint32_t flags;         /* ULY_FLAG_* */
  uint32_t reserved;      /* must be 0 */
} uly_config;

typedef struct uly_plan_s *uly_plan;

/* Validate cfg and build a plan: copies cfg, builds the RoPE angle tables (fp64 on the
 * host, stored fp32 on the device) and a device status word, and looks up the device address
 * of the library's fixed backward scratch (ulysses_attn_bwd_noalloc); with the runtime's
 * default lazy module loading, the first plan on a device is what loads that 64 MiB array
 * there.  No kernel is launched.  Returns ULY_ERR_INVALID_ARG / ULY_ERR_UNSUPPORTED for bad
 * configs, ULY_ERR_OOM or ULY_ERR_CUDA if its buffers cannot be made.  The current CUDA
 * device is the plan's.  A plan does not survive a reset of its device. */
uly_status ulysses_plan(const uly_config *cfg, uly_plan *out);

/* Frees the plan's buffers.  NULL is allowed.  Synchronises the device first. */
uly_status ulysses_plan_destroy(uly_plan plan);

/* Bytes of scratch that ulysses_attn_bwd needs: an fp32 dQ accumulator [P][S][H/P][D],
 * the fp32 row terms Delta [P][H/P][S] and fp16 copies of q, d_o, k and v, each part
 * 256-byte aligned. */
size_t ulysses_workspace_bytes(uly_plan plan);

/* Local QKV projection of every shard (Ulysses-trick page para 2: the projection happens
 * on each rank before any exchange): qkv[s][c] = sum_k x[s][k] * w[c][k], fp32 accumulation,
 * bf16 round-to-nearest-even output.  x [S][hidden], w [C][hidden], qkv [S][C] = the
 * qkv_seq layout.  All ranks share w, so this is one GEMM over all S rows. */
uly_status ulysses_qkv_proj(uly_plan plan, const void *x, const void *w, void *qkv,
                            void *stream);

/* seq->head all-to-all (Ulysses-trick page para 2): for every token s of rank r and
 * column head c, writes q[c/(H/P)][s][c%(H/P)] (query heads), k[..][s][..] and v.
 * in_fp32 != 0: qkv_seq is fp32 and is rounded to bf16 (RNE) on the way.
 * apply_rope != 0 (needs rope_theta > 0): q and k rows are rotated (rotate-half form) by
 * angle s * theta^(-2i/D) for the pair (i, i + D/2), s the global token index, in fp32,
 * then rounded to bf16.  Without RoPE the permutation moves bits unchanged. */
uly_status ulysses_seq_to_head(uly_plan plan, const void *qkv_seq, int in_fp32,
                               int apply_rope, void *q, void *k, void *v, void *stream);

/* seq->head all-to-all of one tensor of n_heads heads (n_heads = H or G; e.g. the
 * upstream gradient dO): x_seq [P][S/P][n_heads][D] -> x_head [P][S][n_heads/P][D]. */
uly_status ulysses_seq_to_head_heads(uly_plan plan, const void *x_seq, int n_heads,
                                     void *x_head, void *stream);

/* Causal GQA attention of every rank's head group over the full sequence (Ulysses-trick
 * page para 2: heads do not interact, so a rank runs ordinary flash attention on the heads
 * it holds; tiled so no S x S matrix is ever stored, Hugging Face post para 3).  For query head
 * h' of rank r (KV head h' / (H/G)):  o = softmax(scale * q k^T, causal) v in bf16 with
 * fp32 softmax and accumulation; lse = natural-log logsumexp of the scaled scores.
 * o_lo (optional, may be NULL; layout of o): receives bf16(O - o), what the bf16 rounding
 * of each output element dropped.  Passing it on to ulysses_attn_bwd lets the backward
 * form its row terms dO.O from O to ~16 significant bits instead of 8. */
uly_status ulysses_attn_fwd(uly_plan plan, const void *q, const void *k, const void *v,
                            void *o, void *o_lo, float *lse, void *stream);

/* Backward of ulysses_attn_fwd for the training step (Hugging Face post para 1: the
 * method is for training).  Inputs q, k, v, o, lse as above, o_lo from the forward (or
 * NULL: the row terms then use the bf16 o alone) and the upstream gradient d_o in head
 * layout [P][S][H/P][D].  Outputs dq [P][S][H/P][D], dk, dv [P][S][G/P][D] in bf16; dk
 * and dv sum the contributions of all query heads of a KV head.
 * The tensor-core operands are fp16 copies of q, k, v and d_o, each multiplied by a power
 * of two chosen per call from the tensor's largest magnitude (and the products P, dS kept
 * in fp16 range), with the inverse powers applied exactly to the outputs.  So gradients as
 * small as a training step's (|d_o| ~ 1e-8) keep fp16's full precision, bf16 inputs above
 * fp16's 65504 are not clipped, and scaling any input by a power of two scales the outputs
 * by exactly that factor (q and k share one exponent, q' = 2^e q and k' = 2^-e k, which
 * balances them and leaves every logit unchanged).  Inputs that no exponent within +-60
 * can bring into fp16's range -- in practice max|q| * max|k| >= 2^30 (logits that large
 * leave a one-hot softmax), or max|v| or max|d_o| beyond about 2^+-60 -- would saturate
 * an fp16 copy; the call then reports ULY_ERR_RANGE through the status word.
 * workspace: ulysses_workspace_bytes(plan) bytes of device memory (fp32 accumulators);
 * its contents on entry do not matter. */
uly_status ulysses_attn_bwd(uly_plan plan, const void *q, const void *k, const void *v,
                            const void *o, const void *o_lo, const float *lse,
                            const void *d_o, void *dq, void *dk, void *dv, void *workspace,
                            void *stream);

/* ulysses_attn_bwd without a caller-provided workspace.  The pages have no counterpart:
 * this serves callers that cannot allocate device memory at call time -- a program that
 * has handed all of HBM to its own pool or caching allocator, a latency-critical path
 * that must not pay cudaMalloc's implicit synchronisation, a plain C caller without a
 * device allocator.  Same arguments and results as ulysses_attn_bwd (minus workspace).
 * The scratch is a fixed 64 MiB array inside the library's device memory.  A GPU holds it
 * from the first ulysses_plan made on it (with eager module loading: from the library's
 * load) until the process exits; ulysses_plan looks its address up, so no call of this
 * entry point, its first included, allocates or loads anything.  Plans whose backward
 * needs more scratch (ulysses_workspace_bytes) get ULY_ERR_UNSUPPORTED and nothing is
 * launched.  All calls share the array: calls that may overlap on the GPU race, so order
 * them (e.g. one stream).  The plan's device must be the current device. */
uly_status ulysses_attn_bwd_noalloc(uly_plan plan, const void *q, const void *k,
                                    const void *v, const void *o, const void *o_lo,
                                    const float *lse, const void *d_o, void *dq, void *dk,
                                    void *dv, void *stream);

/* head->seq all-to-all, the inverse of seq->head (Hugging Face post para 5: a second
 * exchange undoes the first and brings back the sequence sharding): x_head [P][S][n_heads/P][D] ->
 * x_seq [P][S/P][n_heads][D].  n_heads = H for o and dq, G for dk and dv. */
uly_status ulysses_head_to_seq(uly_plan plan, const void *x_head, int n_heads, void *x_seq,
                               void *stream);

/* Rest of the block's training step (the method is for training: "Ulysses Sequence
 * Parallelism: Training with Million-Token Contexts" para 1; these gradients mirror the
 * forward steps above in reverse).
 *
 * head->seq all-to-all of the attention gradients back into the projection layout:
 * dq [P][S][H/P][D], dk, dv [P][S][G/P][D] -> dqkv_seq [P][S/P][H + 2G][D] (= [S][C]),
 * the exact inverse of ulysses_seq_to_head's permutation.  apply_rope != 0 (needs
 * rope_theta > 0) applies the RoPE backward to the q and k parts: each pair (i, i + D/2)
 * at global position s is turned back by s * theta^(-2i/D) (the transpose of the forward
 * rotation), in fp32, rounded once to bf16.  Without RoPE it moves bits unchanged. */
uly_status ulysses_head_to_seq_qkv(uly_plan plan, const void *dq, const void *dk,
                                   const void *dv, int apply_rope, void *dqkv_seq,
                                   void *stream);

/* Backward of ulysses_qkv_proj: dx[s][k] = sum_c dqkv[s][c] w[c][k] (bf16 [S][hidden], RNE)
 * and dw[c][k] = sum_s dqkv[s][c] x[s][k] (fp32 [C][hidden], summed over all S tokens of
 * all shards, as the shared weight's gradient); fp32 accumulation.  Either output may be
 * NULL to skip it. */
uly_status ulysses_qkv_proj_bwd(uly_plan plan, const void *x, const void *w,
                                const void *dqkv, void *dx, float *dw, void *stream);

/* Output projection of the block, fused with the head->seq all-to-all of O ("Snowflake's
 * Ulysses trick ...", para 2: the inverse all-to-all restores the sequence sharding, after
 * which the block's output projection runs on each rank's tokens):
 *   y[s][j] = sum_{h,d} o_seq[s][h][d] * wo[j][h*D + d]
 * read straight from the attention's head layout o_head [P][S][H/P][D] (bf16), so O is never
 * stored in the sequence layout.  wo: bf16 [hidden][H*D] (nn.Linear layout).  y: bf16
 * [S][hidden] (= [P][S/P][hidden]), fp32 accumulation, round to nearest even. */
uly_status ulysses_o_proj(uly_plan plan, const void *o_head, const void *wo, void *y,
                          void *stream);

/* Backward of ulysses_o_proj, fused with the seq->head all-to-all of dO:
 *   do_head (bf16, head layout [P][S][H/P][D]) = dy wo, written straight in the layout
 *     ulysses_attn_bwd reads;
 *   dwo (fp32 [hidden][H*D]) = dy^T o_seq, summed over all S tokens of all shards.
 * dy: bf16 [S][hidden].  Either output may be NULL to skip it. */
uly_status ulysses_o_proj_bwd(uly_plan plan, const void *o_head, const void *wo,
                              const void *dy, void *do_head, float *dwo, void *stream);

/* Synchronises `stream`, reads the plan's device status word, clears it and returns it
 * (ULY_OK, or e.g. ULY_ERR_TIMEOUT, ULY_ERR_RANGE).  ULY_ERR_CUDA if the synchronisation
 * itself fails.  Until it is called after a device-side failure, the plan's later calls
 * abort early (see the conventions above). */
uly_status ulysses_sync_status(uly_plan plan, void *stream);

/* Bytes read plus written by this plan's permute kernels since it was made: what the
 * all-to-all kernels move through HBM. */
uint64_t ulysses_bytes_moved(uly_plan plan);

/* Per-rank all-to-all volume of one block (Ulysses-trick page para 3): the bytes one
 * rank sends to other ranks in the seq->head exchange ((S/P) * (H + 2G) * D * 2 *
 * (P-1)/P) and in the head->seq exchange ((S/P) * H * D * 2 * (P-1)/P). */
uly_status ulysses_a2a_volume(const uly_config *cfg, uint64_t *seq_to_head_bytes,
                              uint64_t *head_to_seq_bytes);

/* Ring attention, the comparator the Ulysses-trick page sets against (para 3: its per-GPU
 * volume is O(hidden * S), against Ulysses' O(hidden * S / P)), run on the same virtual
 * ranks so that its exchange and its time can be measured beside the all-to-alls.
 *
 * The sequence stays sharded: q_seq [P][S/P][H][D], k_seq, v_seq [P][S/P][G][D] (bf16; rank
 * r holds tokens [r*S/P, (r+1)*S/P), RoPE already applied by the caller).  In step
 * t = 0 .. P-1 every rank r attends its queries to the K/V shard it holds, (r - t) mod P,
 * with the causal mask on global positions, and merges the result into its running softmax
 * state; then every rank passes the shard it holds to rank r + 1 (a device copy: the
 * ring's communication).  Output o_seq [P][S/P][H][D] (bf16) and lse [P][H][S/P] (fp32,
 * natural log) equal causal attention of the whole sequence.
 * workspace: ulysses_ring_workspace_bytes(plan) bytes of device memory (two K/V ring
 * buffers and the fp32 running state); contents on entry do not matter.
 * Every launch adds the exchange's read + write bytes to ulysses_bytes_moved. */
size_t ulysses_ring_workspace_bytes(uly_plan plan);
uly_status ulysses_ring_attn_fwd(uly_plan plan, const void *q_seq, const void *k_seq,
                                 const void *v_seq, void *o_seq, float *lse, void *workspace,
                                 void *stream);

/* Per-rank volume of ring attention's forward: the bytes one rank sends, its K/V shard
 * forwarded P - 1 times: (P-1) * (S/P) * 2G * D * 2. */
uly_status ulysses_ring_volume(const uly_config *cfg, uint64_t *bytes);

/* ---------------------------------------------------------------- real ranks (GPUs)
 * The same block on P GPUs, one process (rank) per GPU, as "Snowflake's Ulysses trick
 * ..." para 2 describes it: the two all-to-alls cross GPUs.  A rank plan describes rank
 * `rank` of the group (cfg->P = the number of ranks): it holds the rank's token shard
 * (n = S/P tokens from rank*n on) and, after the first exchange, the whole sequence for its
 * head group (hl = H/P query heads, gl = G/P KV heads).  Layouts on one rank:
 *   x_local        [n][hidden]             the shard's rows of x
 *   qkv_local      [n][H + 2G][D]          its projection (= [n][C])
 *   send_q         [P][n][hl][D]           block p goes to rank p: the shard's rows of rank
 *   send_k, send_v [P][n][gl][D]           p's head group (RoPE applied at global positions)
 *   q (received)   [P][n][hl][D]           block p came from rank p: p's shard of this head
 *                  = [S][hl][D]            group -- in token order, the attention's layout
 *   k, v           [S][gl][D]
 *   o, do_head     [S][hl][D] = [P][n][hl][D]   sent as is: block p holds rank p's tokens
 *   lse            [hl][S]                 fp32
 *   o (received)   [P][n][hl][D]           block p came from rank p: its heads of this shard
 *   o_local        [n][H][D]
 * The calls that accept a rank plan:
 *   ulysses_qkv_proj, ulysses_qkv_proj_bwd   on the shard's n rows (dw sums this rank's
 *                     tokens only: the caller sums it over the ranks, as for any weight
 *                     that data-parallel ranks share)
 *   ulysses_a2a_pack_qkv, ulysses_a2a_pack_heads       write send buffers
 *   ulysses_a2a_exchange                               the all-to-all itself
 *   ulysses_a2a_unpack_heads, ulysses_a2a_unpack_qkv   read receive buffers
 *   ulysses_attn_fwd, ulysses_attn_bwd, ulysses_attn_bwd_noalloc, ulysses_workspace_bytes
 *                     the head group over all S tokens (q, k, v, o, lse as above)
 *   ulysses_o_proj    reads o's receive buffer [P][n][hl][D] directly (no unpack)
 *   ulysses_o_proj_bwd  writes do_head as dO's send buffer [P][n][hl][D] directly
 * The single-GPU permutes (ulysses_seq_to_head, ulysses_seq_to_head_heads,
 * ulysses_head_to_seq, ulysses_head_to_seq_qkv) and ring attention reject a rank plan
 * with ULY_ERR_INVALID_ARG.  No kernel ever reads another GPU's memory: every exchange
 * lands in the receiving rank's own buffers before any kernel reads it. */
uly_status ulysses_plan_rank(const uly_config *cfg, int32_t rank, uly_plan *out);

/* One block of an all-to-all, seen from `rank`: what it sends to `peer` and what it
 * receives from `peer`.  Offsets and counts are in elements (D per head row). */
typedef struct uly_a2a_block {
  int32_t peer;
  int32_t n_tokens;          /* tokens in the block: S/P */
  int32_t n_heads;           /* heads in the block: n_heads/P */
  int32_t reserved;
  int64_t send_token_begin;  /* global index of the first token sent to peer */
  int64_t recv_token_begin;  /* global index of the first token received from peer */
  int32_t send_head_begin;   /* global index of the first head sent to peer */
  int32_t recv_head_begin;   /* global index of the first head received from peer */
  uint64_t send_offset;      /* where the block starts in the send buffer */
  uint64_t recv_offset;      /* where the block starts in the receive buffer */
  uint64_t count;            /* elements in the block: n_tokens * n_heads * D */
} uly_a2a_block;

/* The all-to-all's block table of `rank` (host only, no GPU needed): blocks[p] for every
 * peer p = 0 .. P-1 (p = rank is the block a rank keeps).  to_head != 0: seq->head of a
 * tensor of n_heads heads (H, or G for k and v): rank r sends its tokens' heads
 * [p*n_heads/P, (p+1)*n_heads/P) to p and receives p's tokens of its own heads.  to_head
 * == 0: head->seq, the inverse.  Both buffers are block-major ([P][n][n_heads/P][D]), so
 * every block is one contiguous run and all blocks have the same size. */
uly_status ulysses_a2a_table(const uly_config *cfg, int32_t rank, int32_t to_head,
                             int32_t n_heads, uly_a2a_block *blocks);

/* seq->head send buffers of a rank (rank plans only): qkv_local [n][H + 2G][D] (bf16, or
 * fp32 when in_fp32, rounded to bf16 on the way) -> send_q [P][n][hl][D], send_k, send_v
 * [P][n][gl][D].  apply_rope != 0 (needs rope_theta > 0) rotates q and k as
 * ulysses_seq_to_head does, at the tokens' global positions rank*n + t. */
uly_status ulysses_a2a_pack_qkv(uly_plan plan, const void *qkv_local, int in_fp32,
                                int apply_rope, void *send_q, void *send_k, void *send_v,
                                void *stream);

/* seq->head send buffer of one tensor of n_heads heads (e.g. dO): x_local [n][n_heads][D]
 * -> send [P][n][n_heads/P][D] (rank plans only). */
uly_status ulysses_a2a_pack_heads(uly_plan plan, const void *x_local, int n_heads, void *send,
                                  void *stream);

/* head->seq receive buffer of one tensor of n_heads heads (e.g. o): recv
 * [P][n][n_heads/P][D] -> x_local [n][n_heads][D] (rank plans only). */
uly_status ulysses_a2a_unpack_heads(uly_plan plan, const void *recv, int n_heads,
                                    void *x_local, void *stream);

/* head->seq receive buffers of the attention gradients (rank plans only): recv_dq
 * [P][n][hl][D], recv_dk, recv_dv [P][n][gl][D] -> dqkv_local [n][H + 2G][D], with the RoPE
 * backward on the q and k parts at the global positions when apply_rope != 0, as
 * ulysses_head_to_seq_qkv does. */
uly_status ulysses_a2a_unpack_qkv(uly_plan plan, const void *recv_dq, const void *recv_dk,
                                  const void *recv_dv, int apply_rope, void *dqkv_local,
                                  void *stream);

/* The all-to-all between the ranks of a rank plan's group, over NCCL (the library loads
 * libnccl.so.2 when first needed; ULY_ERR_UNSUPPORTED if it cannot).  For each of the
 * n_buffers (1..8) buffer pairs, rank r sends bytes_per_peer[i] bytes from
 * send[i] + p * bytes_per_peer[i] to every rank p and receives p's block into
 * recv[i] + p * bytes_per_peer[i] -- the block-major layout of ulysses_a2a_table.  All
 * sends and receives form one NCCL group, enqueued on `stream`.  comm must be an NCCL
 * communicator (ncclComm_t) of exactly the plan's P ranks in which this process is rank
 * `rank` (ulysses_nccl_comm_init makes one).  Send and receive buffers are device memory
 * of this GPU and must not overlap. */
uly_status ulysses_a2a_exchange(uly_plan plan, void *comm, int32_t n_buffers,
                                const void *const *send, void *const *recv,
                                const uint64_t *bytes_per_peer, void *stream);

/* NCCL set-up for ulysses_a2a_exchange, so that a plain C caller needs no NCCL header:
 * one rank draws the 128-byte id, every rank receives it (by any channel) and joins with
 * its rank.  ulysses_nccl_comm_init must be called by all nranks processes, each with its
 * own GPU current; it blocks until all have joined. */
uly_status ulysses_nccl_unique_id(uint8_t id[128]);
uly_status ulysses_nccl_comm_init(int32_t nranks, int32_t rank, const uint8_t id[128],
                                  void **comm);
uly_status ulysses_nccl_comm_destroy(void *comm);

/* Description of the last error on this thread ("" if none). */
const char *ulysses_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H_ */
