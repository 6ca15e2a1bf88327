/*
 * sd_verify.h — C ABI of the GB300 speculative-decoding verify library.
 *
 * The library implements the verify step of speculative decoding and the
 * outcome prediction of speculative speculative decoding as hand-written
 * CUDA kernels for sm_103a.  Every entry point is stream-ordered and
 * asynchronous: it validates its arguments on the host, enqueues kernels on
 * the caller's stream and returns without synchronising.  All pointers that
 * are not marked "host" are device pointers owned by the caller; the library
 * allocates no memory and keeps no pointer after a call returns.
 *
 * Sources of the method (web pages):
 *  - "What is speculative decoding" explainer (lotook.com), section on the
 *    four-stage loop: draft K tokens recording each position's
 *    distribution, score all positions in one target pass, accept/reject
 *    left to right (greedy: match the target's top choice; sampling: keep a
 *    token the target rates at least as high as the draft, else keep it
 *    with the target/draft probability ratio), resample the first rejected
 *    position from a residual of both distributions, or take a bonus token
 *    from position K+1 when all K are accepted; FAQ on losslessness.
 *  - "Speculative Speculative Decoding" blog (jiwasawa.github.io), section
 *    "Saguaro 1. Outcome Prediction": predict the verify outcome
 *    (accept length, bonus token) from the draft logits' top tokens with a
 *    fan-out per position, cache pre-speculations under those keys.
 *  - "LLMの生成を5倍速くする「D3D」を図で読む" (animemo.app), sections
 *    検証のしくみ③ and 検証のまとめ (greedy worked example, accept length
 *    tau), 答え:ありうる結果すべてに、先回りして下書きする (the drafter's own
 *    next candidates for each rejection position plus one all-accepted
 *    key), ヒット / ミス (hit test).
 *
 * Readings where the pages are silent (the exact formulas are not printed):
 *  - temperature T enters as softmax(logits / T); T == 0 is greedy;
 *  - accept d_j iff u_j <= p_j(d_j) / q_j(d_j), u_j in (0,1];
 *  - residual w_i = max(0, p_i - q_i) sampled by inverse CDF in index order
 *    (the smallest i whose running sum exceeds u * sum(w)); if the residual
 *    is identically zero the draw falls back to p;
 *  - uniforms: Philox4x32-10 keyed by the 64-bit seed, counter
 *    (row, position, slot, 0), word 0 -> u = ((x >> 8) + 1) * 2^-24;
 *    slot 0 = accept test, slot 1 = residual or bonus draw; the row number
 *    is row_base + b so that a batch split over devices draws the same
 *    uniforms;
 *  - greedy ties go to the lowest index.
 */
#ifndef SD_VERIFY_H_
#define SD_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side return codes. */
typedef enum {
  SD_OK = 0,
  SD_ERR_INVALID_ARG = 1, /* a null pointer, a size out of range, a bad dtype */
  SD_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement  */
  SD_ERR_CUDA = 3         /* the CUDA runtime reported an error at launch    */
} sd_status_t;

/* Device-side status bits, OR-ed into the optional *status word.  Kernels
 * never trap and never wait on one another: a data error marks the affected
 * row invalid (tau = 0, all out_tokens = -1, num_accepted = 0, hit = 0) and
 * sets a bit here. */
#define SD_STATUS_BAD_TOKEN 0x1u /* a draft token outside [0, V)              */
#define SD_STATUS_BAD_TEMP 0x2u  /* a temperature < 0, NaN or infinite        */
#define SD_STATUS_NONFINITE 0x4u /* with SD_FLAG_CHECK_FINITE: a row the call
                                    read holds NaN or +inf, or only -inf      */

typedef enum { SD_F32 = 0, SD_BF16 = 1 } sd_dtype_t;

/* Limits of this build. */
#define SD_MAX_K 32         /* draft tokens per row                           */
#define SD_MAX_V 262144     /* vocabulary size                                */
#define SD_MAX_FANOUT 8     /* outcome-prediction candidates per position     */

/* sd_verify flags */
#define SD_FLAG_PREDICT 0x1u /* also build the outcome-prediction keys from
                                the draft rows read by this pass (keys_out)  */
#define SD_FLAG_COMPACT 0x2u /* also pack the emitted tokens of all rows
                                (offsets, packed), as sd_compact does         */
#define SD_FLAG_CHECK_FINITE 0x4u /* check every logit row the call reads for
                                a sequence (its K+1 target rows; draft row j
                                when the sequence is sampled or keys are built
                                at j; the bonus draft row when keys are built
                                at K): a NaN or +inf, or a row of only -inf,
                                makes the sequence invalid and sets
                                SD_STATUS_NONFINITE (single -inf values are
                                valid logits of weight 0).  Without the flag
                                such rows give unspecified tokens (no fault).
                                The keys of a flagged sequence are unspecified. */

/*
 * Arguments of sd_verify.  Logits are contiguous, row-major, last dimension V,
 * in the dtype given; a row need not start on any particular alignment.
 */
typedef struct sd_verify_args {
  int32_t B;            /* rows (sequences) in the batch, >= 0               */
  int32_t K;            /* draft tokens per row, 0 <= K <= SD_MAX_K          */
  int32_t V;            /* vocabulary size, 1 <= V <= SD_MAX_V               */
  sd_dtype_t dtype;     /* SD_F32 or SD_BF16                                  */
  uint32_t flags;       /* SD_FLAG_*                                          */
  uint64_t seed;        /* key of the uniforms (one per verify round)        */
  int64_t row_base;     /* global number of row 0 (uniform counters)         */

  const void *target_logits;   /* [B][K+1][V]  required                      */
  const void *draft_logits;    /* [B][K][V]    required when K > 0           */
  const int32_t *draft_tokens; /* [B][K]       required when K > 0           */
  const float *temperature;    /* [B]          required; 0 => greedy row     */

  /* Outcome-prediction keys to test the outcome against (optional):
   * [B][n_keys][2] pairs (position, token) as written by sd_outcome_predict;
   * (-1,-1) marks an empty slot.  Ignored when SD_FLAG_PREDICT is set. */
  const int32_t *cache_keys;
  int32_t n_keys;

  /* Fused outcome prediction (SD_FLAG_PREDICT): fanout_host [K+1] (host),
   * each 0..SD_MAX_FANOUT; draft_bonus_logits [B][V] optional; keys_out
   * [B][sum(fanout)][2].  The hit test then uses keys_out. */
  const int32_t *fanout_host;
  const void *draft_bonus_logits;
  int32_t *keys_out;

  /* Outputs (required). */
  int32_t *num_accepted; /* [B]                                              */
  int32_t *out_tokens;   /* [B][K+1]: accepted drafts, then the corrected or
                            bonus token, then -1                              */
  int32_t *tau;          /* [B]: num_accepted + 1 (0 for an invalid row)     */

  /* Optional outputs (may be null). */
  uint8_t *hit;          /* [B]: 1 if (num_accepted, emitted token) is a key */
  int32_t *offsets;      /* [B+1] with SD_FLAG_COMPACT: exclusive scan of tau */
  int32_t *packed;       /* [B*(K+1)] with SD_FLAG_COMPACT                    */
  float *accept_ratio;   /* [B][K]: p_j(d_j) / q_j(d_j), sampled rows only    */
  float *p_draft;        /* [B][K]: p_j(d_j), sampled rows only               */
  float *q_draft;        /* [B][K]: q_j(d_j), sampled rows only               */
  int32_t *target_argmax;/* [B][K+1]: top target token per position          */
  int32_t *status;       /* one int32, SD_STATUS_* bits OR-ed in             */

  /* Scratch for the split launch (optional): at least
   * sd_verify_workspace_size(B, K) bytes, 16-byte aligned, caller-owned.
   * With it, the rows of all sequences are streamed by one flat grid that
   * writes per-piece statistics here, and a per-sequence finish reads them
   * back; without it (NULL), one cluster kernel does both on chip.  The
   * contents need no clearing (every record is written before it is read in
   * the same call); calls that share a workspace must not overlap on the GPU
   * (one stream orders them).  Smaller than required: SD_ERR_INVALID_ARG. */
  void *workspace;
  size_t workspace_bytes;
} sd_verify_args;

/* Bytes of scratch the split launch of sd_verify needs for a batch of B rows
 * of K drafts: (1024 + B (2K + 2)) records of 96 bytes; 0 for arguments out
 * of range. */
size_t sd_verify_workspace_size(int32_t B, int32_t K);

/*
 * The verify step ("What is speculative decoding" explainer (lotook.com),
 * the four-stage loop: stages 2-4, score the K drafted positions in one
 * target pass, accept left to right, resample the first rejection from a
 * residual of both distributions or take the bonus token; "LLMの生成を5倍速く
 * する「D3D」を図で読む" (animemo.app), 検証のしくみ③ and 検証のまとめ: the
 * greedy match, tau = accepted drafts + 1; "Speculative Speculative
 * Decoding" blog (jiwasawa.github.io), Saguaro 1. Outcome Prediction: the
 * keys and the hit test): per-row temperature softmax of the K+1 target and
 * K draft rows, the left-to-right accept/reject scan (argmax match for
 * T == 0), the correction token from the residual at the first rejection or
 * the bonus token from target row K, tau, the optional hit test, and
 * optionally the outcome-prediction keys and the compaction of all rows'
 * tokens.
 * Each logit row is streamed from memory once; the target and draft rows at
 * the first rejection (or target row K) are read a second time for the
 * draw (from L2 when a round's logits fit there).  Two ways to run: with a workspace, a split launch
 * (a streaming launch over the rows of all sequences, every SM moving the
 * same bytes, then a finish launch as its programmatic dependent); without
 * one, a single cluster kernel; plus, with SD_FLAG_COMPACT, a one-CTA
 * packing launch (a programmatic dependent of the last, same stream).
 * Requests outside the split launch's limits
 * (a streaming CTA's share touching more than 2 SD_MAX_K + 2 rows, or B too
 * large for its shared-memory list of sampled rows) take the single launch.
 */
sd_status_t sd_verify(const sd_verify_args *args, void *stream);

/*
 * sd_verify without caller scratch (the pages have no counterpart: this is
 * an interface for callers that cannot allocate device memory when they
 * verify -- a serving runtime whose memory is all handed to its own pool
 * up front, a plugin given only the tensors it works on, a step that must
 * not call an allocator).  Same arguments and results as sd_verify; the
 * workspace fields must be NULL / 0 (else SD_ERR_INVALID_ARG).  The split
 * launch keeps its piece records in a 2 MiB array inside the library
 * (a file-scope __device__ array that every GPU which loads the library
 * holds until the process exits), so sd_verify_workspace_size(B, K) may be
 * at most 2 MiB: 1024 + B (2K + 2) <= 21845 (e.g. B = 256 at K = 32);
 * larger batches return SD_ERR_UNSUPPORTED with a message on stderr.  The
 * call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that
 * first call before capturing a stream into a CUDA graph.  All calls share
 * the one array per device: calls that may overlap on the GPU (other
 * streams, other threads) race on it, so order them on one stream.  The
 * array keeps the last call's records; nothing in it needs clearing, as
 * every record is written before it is read within a call.  Like
 * sd_verify given scratch, it takes the split launch, and the single
 * cluster kernel (which needs no scratch) outside the split launch's
 * limits.  The looked-up address belongs to the device's primary context:
 * it is not valid across cudaDeviceReset (reload the library after one).
 */
sd_status_t sd_verify_noalloc(const sd_verify_args *args, void *stream);

/*
 * Outcome prediction ("Speculative Speculative Decoding" blog
 * (jiwasawa.github.io), Saguaro 1. Outcome Prediction: the likely verify
 * outcomes are the accept lengths paired with the draft's top tokens, with a
 * fan-out per position; "LLMの生成を5倍速くする「D3D」を図で読む"
 * (animemo.app), 答え:ありうる結果すべてに、先回りして下書きする: the
 * drafter's own next candidates at each rejection position plus one
 * all-accepted key): for each row b and position k < K, the fanout[k]
 * tokens with the highest draft logit at k other than the drafted token
 * d_k (ties to the lowest index, -inf logits never chosen), keyed (k, token):
 * the corrections a rejection at k could produce.  For k == K the fanout[K]
 * highest logits of draft_bonus_logits [B][V] (optional; without it those
 * slots stay empty), keyed (K, token): the bonus token when all K are
 * accepted.  keys: [B][n_keys][2], n_keys = sum(fanout); empty slots are
 * (-1,-1).  fanout_host and n_keys_out are host pointers.
 */
sd_status_t sd_outcome_predict(int32_t B, int32_t K, int32_t V, sd_dtype_t dtype,
                               const void *draft_logits, const int32_t *draft_tokens,
                               const void *draft_bonus_logits, const int32_t *fanout_host,
                               int32_t *keys, int32_t *n_keys_out, int32_t *status,
                               void *stream);

/*
 * Vocabulary-sharded verify ("Speculative Speculative Decoding" blog
 * (jiwasawa.github.io), performance and hardware: the target runs on four
 * GPUs, so its logits arrive split over the vocabulary).  S shards cover
 * [0, V) in order; shard `shard` holds columns [v0, v0 + vs) of every logit
 * row: target [B][K+1][vs], draft [B][K][vs], bonus draft [B][vs], each
 * contiguous, on its own device (or all on one device).  The step runs in
 * three calls per shard with an exchange between them:
 *   sd_vshard_stats  -> stats block of this shard (sd_vshard_stats_bytes);
 *                       all-gather the S blocks, in shard order, into
 *                       stats_all;
 *   sd_vshard_mass   -> this shard's mass block (sd_vshard_mass_bytes):
 *                       every shard combines all rows' statistics and takes
 *                       the same accept decisions, then measures its own
 *                       columns' share of the draw, part by part (eight
 *                       column parts per shard); all-gather into mass_all;
 *   sd_vshard_pick   -> outputs: the prefix over the shards' masses names the
 *                       shard holding u * S and the prefix over its parts the
 *                       part; that shard alone scans the part's columns (an
 *                       inverse CDF in levels) and writes the token and the
 *                       hit flag of a sampled row; every shard writes the
 *                       rest, which is the same everywhere.
 * Pre-fill out_tokens with -1 and hit with 0: an element-wise maximum over
 * the shards' outputs (an all-reduce, or on one device running the shards'
 * picks on the same output arrays) completes them.  The results are those of
 * sd_verify on the unsharded logits (num_accepted, out_tokens, tau, hit,
 * keys_out with SD_FLAG_PREDICT), with the same uniforms.  Flags:
 * SD_FLAG_PREDICT (fanout_host, draft_bonus_logits, keys_out),
 * SD_FLAG_CHECK_FINITE.  1 <= S <= 32.  Buffers are caller-owned device
 * memory, 16-byte aligned; nothing in them needs clearing.
 */
typedef struct sd_vshard_args {
  int32_t B, K, V;             /* batch, drafts, full vocabulary              */
  int32_t S, shard;            /* shard count, this shard                     */
  int32_t v0, vs;              /* this shard's columns [v0, v0 + vs)           */
  sd_dtype_t dtype;
  uint32_t flags;
  uint64_t seed;
  int64_t row_base;
  const void *target_logits;   /* [B][K+1][vs]                                */
  const void *draft_logits;    /* [B][K][vs]                                  */
  const int32_t *draft_tokens; /* [B][K], vocabulary ids                      */
  const float *temperature;    /* [B]                                          */
  const int32_t *fanout_host;  /* [K+1] (host), with SD_FLAG_PREDICT          */
  const void *draft_bonus_logits; /* [B][vs] or NULL                          */
  int32_t *keys_out;           /* [B][sum(fanout)][2] (pick)                  */
  int32_t *num_accepted;       /* [B] (pick)                                  */
  int32_t *out_tokens;         /* [B][K+1] (pick), pre-filled with -1        */
  int32_t *tau;                /* [B] (pick)                                  */
  uint8_t *hit;                /* [B] or NULL (pick), pre-filled with 0       */
  int32_t *status;             /* one int32 or NULL                           */
} sd_vshard_args;

size_t sd_vshard_stats_bytes(int32_t B, int32_t K);
size_t sd_vshard_mass_bytes(int32_t B);
sd_status_t sd_vshard_stats(const sd_vshard_args *args, void *stats, void *stream);
sd_status_t sd_vshard_mass(const sd_vshard_args *args, const void *stats_all, void *mass,
                           void *stream);
sd_status_t sd_vshard_pick(const sd_vshard_args *args, const void *stats_all,
                           const void *mass_all, void *stream);

/*
 * The drafter's next pass, packed from the outcome keys ("LLMの生成を5倍速く
 * する「D3D」を図で読む" (animemo.app), sections 答え:ありうる結果すべてに、
 * 先回りして下書きする and パック:24ブロックを1回の計算で).  A block is K+1
 * tokens.  Block 0 is the block under verification: anchor[b] (the last
 * settled token) and the K drafts, at positions anchor_pos[b] + i.  Block
 * 1 + s is the continuation of key s = (k, c) of keys [B][n_keys][2] (as
 * sd_outcome_predict writes them): c at position anchor_pos[b] + 1 + k (the
 * place of the rejected draft k, or the bonus place when k == K), then K
 * copies of mask_token at the following positions; an empty key (-1, -1)
 * or k outside [0, K] gives an empty block (tokens, positions, ctx all -1).
 * ctx[b][blk]: tokens of block 0 that block blk sees besides the shared
 * prefix -- 0 for block 0 (it sees itself), k + 1 for a continuation.
 * Outputs tokens, positions [B][1 + n_keys][K + 1] and ctx [B][1 + n_keys],
 * caller-owned device memory; keys must be 8-byte aligned.  With K = 15
 * and fanout 2 x 11 + 1 this is the pages' 24 blocks x 16 = 384 tokens.
 */
sd_status_t sd_d3d_pack(int32_t B, int32_t K, int32_t n_keys, const int32_t *keys,
                        const int32_t *draft_tokens, const int32_t *anchor,
                        const int32_t *anchor_pos, int32_t mask_token, int32_t *tokens,
                        int32_t *positions, int32_t *ctx, void *stream);

/*
 * N-gram / prompt-lookup drafting ("What is speculative decoding" explainer
 * (lotook.com), FAQ on drafting without a separate model: copy the tokens
 * that follow a span of the prompt and recent output matching the text's
 * ending; "Speculative Speculative Decoding" blog (jiwasawa.github.io),
 * Saguaro fallback: an n-gram model as the light drafter at large batch).
 * Row b's history is history[b][0..lengths[b]) of history [B][L] (int32
 * tokens >= 0, lengths clamped to [0, L]).  For n = n_max down to n_min
 * (1 <= n_min <= n_max <= 16), the last n tokens are looked up at earlier
 * places followed by at least one token; the first n that occurs wins, at
 * its latest occurrence i.  drafts[b][0..K) = the tokens from i + n on (at
 * most up to the end of the history, then -1); count[b] = how many are
 * real; match_pos[b] = i and match_n[b] = n, or -1 / -1 and count 0 when
 * nothing matches.  One CTA per row; L < 2^26.
 */
sd_status_t sd_ngram_draft(int32_t B, int32_t L, int32_t K, int32_t n_max, int32_t n_min,
                           const int32_t *history, const int32_t *lengths, int32_t *drafts,
                           int32_t *count, int32_t *match_pos, int32_t *match_n, void *stream);

/*
 * KV-cache rollback after a round ("What is speculative decoding" explainer
 * (lotook.com), FAQ on speculative decoding and the KV cache: both caches
 * are rolled back and truncated, dropping the rejected drafts' entries).
 * Row b holds kv_len[b] entries in pages of page_size entries listed in
 * block_table [B][max_pages] (in/out); the round appended `appended` of them
 * (K + 1 for the target's verify pass: the anchor and the drafts) and
 * confirms the first tau[b] (as sd_verify writes it; the correction or bonus
 * token has no entry yet).  new_len[b] = before + min(tau, appended, held),
 * before = max(kv_len - appended, 0), held = kv_len - before.  The pages
 * from ceil(new_len / page_size) up to min(ceil(kv_len / page_size),
 * max_pages) are freed: their ids go, row after row, to freed[] (room for
 * B * max_pages ids) at free_offsets[b] (B + 1 entries, the last the total),
 * and their table slots become -1.  One CTA.
 */
sd_status_t sd_kv_rollback(int32_t B, int32_t page_size, int32_t max_pages, int32_t appended,
                           const int32_t *kv_len, const int32_t *tau, int32_t *block_table,
                           int32_t *new_len, int32_t *freed, int32_t *free_offsets,
                           void *stream);

/*
 * Compaction ("What is speculative decoding" explainer (lotook.com), the
 * four-stage loop: the accepted drafts and the resampled or bonus token are
 * appended to the text; "LLMの生成を5倍速くする「D3D」を図で読む"
 * (animemo.app), 検証のまとめ: tau tokens settle per round): offsets[b] =
 * sum of tau over rows before b (B+1 entries) and
 * packed[offsets[b] + i] = out_tokens[b][i] for i < tau[b].  packed needs
 * room for B*(K+1) tokens.  Entries of tau outside [0, K+1] set
 * SD_STATUS_BAD_TOKEN in *status (optional) and count as 0.
 */
sd_status_t sd_compact(int32_t B, int32_t K, const int32_t *out_tokens, const int32_t *tau,
                       int32_t *offsets, int32_t *packed, int32_t *status, void *stream);

/*
 * The uniforms the verify step draws: out[i] = u(seed, row[i], pos[i],
 * slot[i]) as defined above, for n entries (device arrays).  Lets callers
 * reproduce or audit a round.
 */
sd_status_t sd_uniforms(uint64_t seed, int32_t n, const int32_t *row, const int32_t *pos,
                        const int32_t *slot, double *out, void *stream);

/* sizeof(sd_verify_args) as compiled into the library, so that bindings
 * can check their mirror of the struct. */
size_t sd_verify_args_size(void);

/* Version string of the library (static storage). */
const char *sd_version(void);

/* Name of a host-side return code (static storage). */
const char *sd_status_string(sd_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* SD_VERIFY_H_ */
