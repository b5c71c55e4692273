/*
 * dspark.h - C ABI of libdspark: draft-side candidate selection and target-side
 * rejection-sampling verification for DFlash/DSpark block speculative decoding,
 * on one NVIDIA GB300 (sm_103a).
 *
 * Pages this interface follows (cited by title and section):
 *   [G] openvino.genai PR #4847, "Add DSpark and DFlash v2 drafts and sampled drafting
 *       to DFlash speculative decoding" - Description > Change (Markov heads, sampled
 *       drafting), Fixes (split validation windows), Known issues (host argmax), and its
 *       commits on the thresholded top-p filter, the block sampler / candidate selector,
 *       exact sampled speculative decoding, double-precision multinomial sums, the double
 *       uniform, and the d2t checks.
 *   [E] optimum-intel PR #2098, "[OpenVINO] Export DFlash v2 and DSpark drafts for
 *       PagedAttention and continuous batching" - What does this PR do > DFlash v2
 *       (packed Top-K lattice, transitions gated by the draft hidden states).
 *   [P] optimum-intel PR #2099, "[OpenVINO] Support MiniCPM-OCR-1.0-DSpark: DSpark drafts
 *       with a pruned vocabulary" - What does this PR do > Pruned draft vocabulary, Markov
 *       head (top_k = min(64, draft_vocab_size); table zero outside the draft vocabulary).
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless the argument says "host". The caller owns every
 *     buffer; the library allocates nothing except where a function says it uses a
 *     caller-provided workspace `ws` of at least dspark_workspace_size() bytes.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream). Outputs are valid once the stream reaches the call.
 *   - Host-checkable errors (null pointers, sizes, ranges) return before anything is
 *     launched. Errors found on the device are written to `*dev_status` (a device int32
 *     the caller zeroes; the first error wins) and read by the caller after a sync.
 *   - Layouts are row-major. A request r owns block rows row_start[r] + j, j < B, of a
 *     packed row tensor (every block follows at least one context row in [G], so blocks
 *     need not be adjacent); row_start == NULL means row_start[r] = r * B.
 *   - Token ids are int32; d2t offsets are int64 with target id m(i) = i + d2t[i] [P];
 *     d2t == NULL means the identity map (V_t == V_d).
 *   - Ties in any ordering go to the lowest index; -0.0 and +0.0 compare equal.
 *   - Random numbers: Philox4x32-10 keyed by the request's 64-bit seed; counter words
 *     (step mod 2^32, position j, purpose * 2^20 + draw, step >> 32), purpose 0 = draft draw,
 *     1 = acceptance test, 2 = residual or bonus draw; a double uniform takes two output
 *     words: ((x0 >> 5) * 2^26 + (x1 >> 6)) * 2^-53 [G: commit on the double uniform]. The
 *     draft and the verifier take separate seeds [G: exact sampled speculative decoding].
 *   - Softmax weights: z = s / T in float32, w = 2^n P(f) for d = z - zmax >= -64 (t =
 *     fl32(d log2 e), n = rint(t), f = t - n, P the degree-7 Taylor polynomial of 2^f in
 *     float32 FMAs), w = 0 below -64 [G: thresholded top-p commit]; weights are summed in
 *     double [G: double-precision multinomial sums].
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dspark_stream_t; /* identical to cudaStream_t */

typedef enum {
  DSPARK_OK = 0,
  DSPARK_EINVAL = 1,      /* bad argument; nothing was launched */
  DSPARK_ERANGE = 2,      /* a d2t entry maps a draft index outside [0, V_t) */
  DSPARK_EDUP = 3,        /* d2t is not one-to-one where sampled drafting needs it */
  DSPARK_EPROPOSAL = 4,   /* the recorded q of a drafted token is zero */
  DSPARK_ENONFINITE = 5,  /* a row's maximum is not finite */
  DSPARK_ETIMEOUT = 6,    /* a bounded device wait ran out (the kernel returned early) */
  DSPARK_ECUDA = 7,       /* a CUDA runtime call or launch failed */
  DSPARK_EWORKSPACE = 8   /* the workspace is missing, misaligned or too small */
} dspark_status;

typedef enum { DSPARK_BF16 = 0, DSPARK_F32 = 1 } dspark_dtype;

typedef enum {
  DSPARK_MAXSUM = 0, /* max-sum (Viterbi) chain over the K'xK' lattice */
  DSPARK_WALK = 1,   /* greedy walk: best candidate after the token before [G] */
  DSPARK_SAMPLE = 2  /* sampled walk with the request's draft RNG [G] */
} dspark_chain_mode;

typedef enum {
  DSPARK_OP_TOPK = 0,
  DSPARK_OP_LATTICE = 1,
  DSPARK_OP_CHAIN = 2,
  DSPARK_OP_SAMPLE = 3,
  DSPARK_OP_DENSE_WALK = 4,
  DSPARK_OP_VERIFY = 5,
  DSPARK_OP_D2T_CHECK = 6,
  DSPARK_OP_LATTICE_ROW = 7
} dspark_op;

/*
 * Record of the proposal distribution q of drafted tokens [G: exact sampled speculative
 * decoding - the post-filter q each token was drawn from, sparse over the kept tokens or
 * dense, in target ids]. One record row per (request, position); exactly one of the two
 * forms is used (the other form's pointers are NULL).
 *  Sparse: ids[row*cap + k], p[row*cap + k] for k < n[row]: the kept target ids in
 *          ascending draft (or candidate) index order and their renormalised float32 q.
 *  Dense:  z[row*ldz + i] = s_i / T over draft indices i < V_d (float32), zmax[row],
 *          wsum[row] = double sum of the kept weights, and the nucleus cut: index i is
 *          kept iff w_i > wcut[row], or w_i == wcut[row] and i <= icut[row] (w_i > 0
 *          always required). q(i) = kept ? w(z_i - zmax) / wsum : 0.
 */
/*
 * Repetition / presence penalties of a sampled or greedy walk [G: commit on the penalty history -
 * the penalties apply to every token in the history whatever its count; rejected tokens leave it]:
 * ids [R, cap] int32 target ids of each request's history (device), n [R] int32 their number
 * (device); on a candidate whose target id is in the history or was drafted at an earlier position
 * of the block, the walk row entry s becomes s / repetition (s > 0) or s * repetition (s <= 0),
 * then s - presence, in float32. repetition = 1 and presence = 0 leave the rows unchanged.
 */
typedef struct {
  const int32_t* ids;
  const int32_t* n;
  int32_t cap;
  float repetition;
  float presence;
} dspark_penalties;

typedef struct {
  int32_t* ids;
  float* p;
  int32_t* n;
  int32_t cap;
  float* z;
  int64_t ldz;
  float* zmax;
  double* wsum;
  float* wcut;
  int32_t* icut;
} dspark_qrecord;

/* Bytes of workspace `op` needs for R requests x B positions over V columns with K
 * candidates (0: none). Workspaces need 256-byte alignment and no initial contents; calls that
 * share one workspace must not overlap on the GPU. */
size_t dspark_workspace_size(dspark_op op, int64_t R, int32_t B, int64_t V, int32_t K);

/* Human-readable name of a status code (static string). */
const char* dspark_status_string(dspark_status s);

/*
 * d2t validation [G: commit on the d2t checks - one entry per draft logit; the mapping
 * must be one-to-one for sampled drafting, greedy drafting accepts any mapping].
 * d2t[V_d] int64: checks 0 <= i + d2t[i] < V_t for every i (DSPARK_ERANGE) and, when
 * require_injective != 0, that no two draft indices share a target id (DSPARK_EDUP).
 * The verdict goes to *dev_status. ws: dspark_workspace_size(DSPARK_OP_D2T_CHECK, 1, 1,
 * V_t, 0) bytes (a bitmap over the target vocabulary, cleared by the call).
 */
dspark_status dspark_d2t_check(const int64_t* d2t, int64_t V_d, int64_t V_t,
                               int32_t require_injective, void* ws, size_t ws_bytes,
                               int32_t* dev_status, dspark_stream_t stream);

/*
 * d2t validation that allocates nothing: the same checks and verdicts as dspark_d2t_check, for
 * callers that cannot provide a device workspace (runtimes that allocate nothing once serving
 * has started, or hosts whose device memory is owned by another allocator). The pages have no
 * counterpart: this is a library convenience, not part of the method.
 * The duplicate bitmap is a static 128 KB array in the library's device image, so V_t is
 * limited to 1,048,576 target ids; a larger V_t returns DSPARK_EINVAL before any launch.
 * Every call looks up the array's address in the context current at the call (so a device
 * reset or another context is followed); the first call on a device also loads the library's
 * device code there, so make that first call before any stream capture. Every call clears the
 * bitmap on `stream` before use. Calls that overlap on the GPU share the bitmap and race: serialise them (one stream, or
 * events). d2t: device pointer to V_d int64 offsets; *dev_status as for dspark_d2t_check.
 */
dspark_status dspark_d2t_check_noalloc(const int64_t* d2t, int64_t V_d, int64_t V_t,
                                       int32_t require_injective, int32_t* dev_status,
                                       dspark_stream_t stream);

/*
 * Row transform + Top-K + d2t map [G: Change > Markov heads, Top-K candidate scorer;
 * block-sampler commit - rows are backbone logits times the output multiplier, then
 * soft-capped; P: top_k = min(64, draft_vocab_size), target id i + d2t[i]].
 * logits: [rows, ld] of `dtype` (bf16 or float32), V_d <= ld used columns; the block rows of
 *   request r are row_start[r] + j (row_start may be NULL).
 * s_i = l_i * mult; if softcap > 0, s_i = softcap * tanh(s_i / softcap).
 * Outputs, K' = min(K, V_d), 1 <= K <= 64, ordered by (s descending, draft index ascending):
 *   cand_draft [R, B, K'] int32 draft index, cand_tgt [R, B, K'] int32 target id (-1 and
 *   DSPARK_ERANGE on *dev_status when a chosen index maps outside [0, V_t)), cand_val
 *   [R, B, K'] float32 s.
 * Needs no workspace: each row is selected by one thread block streaming it once.
 */
dspark_status dspark_topk(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                          int64_t V_d, int64_t ld, const int64_t* row_start, int32_t K,
                          float mult, float softcap, const int64_t* d2t, int64_t V_t,
                          int32_t* cand_draft, int32_t* cand_tgt, float* cand_val,
                          int32_t* dev_status, dspark_stream_t stream);

/*
 * Markov-head transition lattice [G: Change > Markov heads - the scorer rates the K best
 * candidates of neighbouring positions; E: DFlash v2 - packed Top-K lattice gated by the
 * draft hidden states; P: Markov head - the next-token table lives over the target
 * vocabulary]. Head form: tau(a, b) = E[a] . W[b], E and W [V_t, rank] row-major in
 * `table_dtype`; gate gamma_{r,j} = sigmoid(h_{r,j} . g) with h the hidden row of block
 * row (r, j) ([rows, ldh], `hidden_dtype`) and g [H]; gamma = 1 when hidden == NULL.
 *   trans[r, 0, 0, b]  = gamma_{r,0} tau(prev[r], cand_tgt[r,0,b]),  trans[r,0,a>0,:] = 0;
 *   trans[r, j, a, b]  = gamma_{r,j} tau(cand_tgt[r,j-1,a], cand_tgt[r,j,b]),  j >= 1;
 *   gate[r, j] = gamma_{r,j}.
 * cand_tgt [R, B, K] int32 (K = K' of dspark_topk, 1..64); prev [R] int32 target ids.
 * trans [R, B, K, K] float32, gate [R, B] float32. bf16 tables with rank % 64 == 0 and
 * rank <= 512 use the tensor cores (tcgen05); other tables use CUDA-core FMAs.
 * Out-of-range ids set DSPARK_ERANGE and give zero transitions.
 */
dspark_status dspark_lattice_score(const int32_t* cand_tgt, const int32_t* prev, int64_t R,
                                   int32_t B, int32_t K, const void* E, const void* W,
                                   dspark_dtype table_dtype, int64_t V_t, int32_t rank,
                                   const void* hidden, const void* g, dspark_dtype hidden_dtype,
                                   int32_t H, int64_t ldh, const int64_t* row_start,
                                   float* trans, float* gate, int32_t* dev_status,
                                   dspark_stream_t stream);

/*
 * Chain selection over the lattice [G: block-sampler commit - greedy requests walk the
 * lattice taking the best candidate after the token before; sampled requests walk it
 * with the draft RNG]. Unary scores u = cand_val [R, B, K], transitions trans
 * [R, B, K, K] as written by dspark_lattice_score, all float32.
 *   DSPARK_MAXSUM: delta_0 = u_0 + A_0[0]; delta_j[b] = u_j[b] + max_a(delta_{j-1}[a] +
 *     A_j[a, b]) (lowest a on ties); the chain ends at argmax delta_{B-1}; score = its max.
 *   DSPARK_WALK: b_j = argmax_b fl32(u_j[b] + A_j[b_{j-1}, b]) (A_0 row 0 for j = 0).
 *   DSPARK_SAMPLE: the same row, sampled at `temperature`/`top_p` over the K candidates
 *     (candidate rank is the index), uniform U(seed[r], step[r], j, purpose 0); the sparse
 *     q of every position goes to q->ids/p/n with q->cap >= K. temperature <= 0 is greedy.
 *     min_p in [0, 1] (0: off) [G: commit on the thresholded filters - MinPFilter]: after top-p,
 *     only candidates whose probability is at least min_p times the top candidate's are kept.
 * Mixed batches [G: Change > Sampled drafting - greedy and sampled requests share one
 * continuous-batching step]: temperature_r / top_p_r, when not NULL, are [R] float32 device
 * arrays of per-request values that replace the scalars in DSPARK_SAMPLE (a request with
 * temperature <= 0 walks greedily and records q = 1 on its token), and so does min_p_r for min_p;
 * a NaN temperature, a top_p <= 0 or a min_p outside [0, 1] there sets DSPARK_EINVAL on
 * *dev_status and walks that request greedily.
 * penalties: NULL, or the repetition/presence penalties of DSPARK_WALK and DSPARK_SAMPLE
 * (DSPARK_EINVAL with DSPARK_MAXSUM: the penalty of a row depends on the path before it).
 * Outputs: chain_rank [R, B] int32, chain_tgt [R, B] int32 (= cand_tgt at the rank),
 * score [R] float32 (sum of the chosen, penalized row entries; the max for MAXSUM).
 * seed, step: [R] uint64 (SAMPLE with a sampled request). No workspace.
 */
dspark_status dspark_chain_select(const float* cand_val, const float* trans,
                                  const int32_t* cand_tgt, int64_t R, int32_t B, int32_t K,
                                  dspark_chain_mode mode, float temperature, float top_p,
                                  float min_p, const float* temperature_r, const float* top_p_r,
                                  const float* min_p_r, const dspark_penalties* penalties,
                                  const uint64_t* seed, const uint64_t* step,
                                  int32_t* chain_rank, int32_t* chain_tgt, float* score,
                                  const dspark_qrecord* q, int32_t* dev_status,
                                  dspark_stream_t stream);

/*
 * Lattice and greedy chain in one call [G: Change > Markov heads, block-sampler commit; E:
 * DFlash v2 packed Top-K lattice]: the same results as dspark_lattice_score followed by
 * dspark_chain_select with mode DSPARK_MAXSUM or DSPARK_WALK (arguments as there). For bf16
 * tables with rank % 64 == 0, rank <= 512 and B <= 8 it is one launch: the B tiles of a
 * request are one thread-block cluster and the chain is decided on chip, so trans and gate
 * may be NULL (not written). Otherwise it runs the two calls and trans must not be NULL.
 */
dspark_status dspark_lattice_chain(const float* cand_val, const int32_t* cand_tgt, const int32_t* prev,
                                   int64_t R, int32_t B, int32_t K, const void* E, const void* W,
                                   dspark_dtype table_dtype, int64_t V_t, int32_t rank,
                                   const void* hidden, const void* g, dspark_dtype hidden_dtype,
                                   int32_t H, int64_t ldh, const int64_t* row_start,
                                   dspark_chain_mode mode, float* trans, float* gate,
                                   int32_t* chain_rank, int32_t* chain_tgt, float* score,
                                   int32_t* dev_status, dspark_stream_t stream);

/*
 * Full-row multinomial drafting without a head [G: Change > Sampled drafting; commits on
 * the thresholded top-p filter, double sums and the double uniform]. Rows as in
 * dspark_topk (transform included). Per block row (r, j): z = s / T, weights, top-p
 * nucleus (shortest prefix of (w desc, index asc) whose double mass exceeds top_p), draw
 * with U(seed[r], step[r], j, purpose 0) walking kept indices in ascending order.
 * temperature <= 0: argmax. out_tgt [R, B] int32 target ids, out_idx [R, B] int32 draft
 * indices (nullable). q: NULL, or a record (sparse with cap >= the nucleus size, else
 * DSPARK_EINVAL on *dev_status and n = -1; or dense with ldz >= V_d). ws: optional device
 * scratch; with at least dspark_workspace_size(DSPARK_OP_SAMPLE, R, B, V_d, 0) bytes (one row of
 * V_d floats per SM, 16-byte aligned) the top-p rows keep their weights there between the nucleus
 * passes instead of recomputing them; smaller or NULL: recomputed, same results.
 * min_p in [0, 1] (0: off) [G: commit on the thresholded filters - MinPFilter]: after the
 * nucleus, only indices whose probability is at least min_p times the top one's are kept (the
 * weight test w >= min_p); where that cuts inside the nucleus, a dense record's cut is
 * (wcut, icut) = (min_p, 0x7FFFFFFF).
 * Mixed batches: temperature_r / top_p_r / min_p_r, when not NULL, are [R] float32 device arrays
 * of per-request values replacing the scalars (temperature <= 0: that request's rows take the
 * argmax); a NaN temperature, top_p <= 0 or min_p outside [0, 1] there sets DSPARK_EINVAL and
 * takes the argmax.
 */
dspark_status dspark_sample(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                            int64_t V_d, int64_t ld, const int64_t* row_start,
                            const int64_t* d2t, int64_t V_t, float mult, float softcap,
                            float temperature, float top_p, float min_p, const float* temperature_r,
                            const float* top_p_r, const float* min_p_r, const uint64_t* seed,
                            const uint64_t* step, int32_t* out_tgt, int32_t* out_idx,
                            const dspark_qrecord* q, void* ws, size_t ws_bytes,
                            int32_t* dev_status, dspark_stream_t stream);

/*
 * Dense Markov walk, markov_head_top_k = 0 [G: Change > Markov heads - the dense walk
 * corrects every drafted position with one head inference per position; block-sampler
 * commit - a dense step biases the scaled rows by the token drafted before].
 * For j = 0..B-1, per request: v_j[i] = s_j[i] + gamma_j tau(prev_j, m(i)) over draft
 * indices i < V_d; x_j = argmax (temperature <= 0) or a draw as in dspark_sample with
 * U(seed[r], step[r], j, purpose 0); out_tgt[r, j] = m(x_j) = prev_{j+1}; prev_0 = prev[r].
 * Head and gate arguments as in dspark_lattice_score (bf16 tables, rank % 64 == 0, rank
 * <= 256, use the tensor cores). q: NULL or a dense record (ldz >= V_d). R <= 128.
 * ws: dspark_workspace_size(DSPARK_OP_DENSE_WALK, R, B, V_d, 0).
 */
dspark_status dspark_dense_walk(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                                int64_t V_d, int64_t ld, const int64_t* row_start,
                                const int32_t* prev, const void* E, const void* W,
                                dspark_dtype table_dtype, int32_t rank, int64_t V_t,
                                const int64_t* d2t, const void* hidden, const void* g,
                                dspark_dtype hidden_dtype, int32_t H, int64_t ldh, float mult,
                                float softcap, float temperature, float top_p,
                                const uint64_t* seed, const uint64_t* step, int32_t* out_tgt,
                                int32_t* out_idx, const dspark_qrecord* q, void* ws,
                                size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream);

/*
 * Rejection-sampling verification [G: commit on exact sampled speculative decoding -
 * accept with probability min(1, p/q), otherwise emit a draw from norm(max(0, p - q)) and
 * drop the later candidates; accepted tokens report the target's log-probability; ids
 * beyond a model's row have zero probability; q is recorded in target ids, sparse or dense;
 * Fixes > split validation windows - row j validates candidate j, row n is the bonus row].
 * tgt_logits: [rows, ld] of `dtype`; request r owns rows row_start[r] + j, j <= B (B + 1
 * rows; row_start NULL means r * (B + 1)). draft_tgt [R, B] int32 target ids, n_draft [R]
 * int32 in 0..B; a request whose n is outside 0..B gets n_accepted = -1 and every
 * out_tokens entry -1, with DSPARK_EINVAL on *dev_status (nothing of it is indexed).
 * q: the proposal record of the drafted tokens, one record row per (r, j) at r * B + j:
 *   sparse - ids in target space, any number of entries up to cap per row;
 *   dense  - over record indices i < V_q (the record's width). With q_d2t == NULL index i
 *            is target id i (ids >= V_q have q = 0); with q_d2t (int64 [V_q], one-to-one)
 *            index i is target id i + q_d2t[i] (a pruned draft vocabulary), and target ids
 *            outside its image have q = 0. q_d2t must be NULL for a sparse record.
 * q is ignored when temperature <= 0.
 * p_j is the post-filter target distribution at (temperature, top_p). For j < n: accept
 * iff U(vseed[r], step[r], j, 1) < p_j(x_j)/q_j(x_j) (double); first rejection: emit a
 * draw from norm(max(0, p_j - q_j)) with U(..., j, 2) and stop; all accepted: bonus draw
 * from p_n with U(..., n, 2). temperature <= 0: accept iff x_j == argmax p_j, emit argmax.
 * Outputs: out_tokens [R, B+1] (accepted tokens then the correction or bonus; -1 after),
 * n_accepted [R] (-1 with DSPARK_EPROPOSAL when the first position that is not accepted has
 * q(x_j) = 0), logprob [R, B+1] float32 (log p_j of each emitted token; greedy reports the
 * temperature-1 log-probability).
 * ws: dspark_workspace_size(DSPARK_OP_VERIFY, R, B, V_t, 0).
 * Mixed batches [G: Description > Fixes > Split validation windows; Change > Sampled drafting]:
 * temperature_r / top_p_r, when not NULL, are [R] float32 device arrays of per-request values
 * replacing the scalars; a request with temperature <= 0 (or NaN) is verified greedily (argmax
 * matching, temperature-1 log-probabilities), the others by the rejection test with their own
 * temperature and top_p; q, vseed and step are then required. A top_p <= 0 there sets
 * DSPARK_EINVAL and verifies that request without a nucleus. n_draft < B validates a prefix.
 * min_p (and min_p_r per request) in [0, 1]: the target's post-filter p keeps, after top-p, only
 * the ids whose probability is at least min_p times the top id's, as the draft's filters did.
 */
dspark_status dspark_verify(const void* tgt_logits, dspark_dtype dtype, int64_t R, int32_t B,
                            int64_t V_t, int64_t ld, const int64_t* row_start,
                            const int32_t* draft_tgt, const int32_t* n_draft,
                            const dspark_qrecord* q, int64_t V_q, const int64_t* q_d2t,
                            float temperature, float top_p, float min_p, const float* temperature_r,
                            const float* top_p_r, const float* min_p_r, const uint64_t* vseed,
                            const uint64_t* step, int32_t* out_tokens, int32_t* n_accepted,
                            float* logprob, void* ws, size_t ws_bytes, int32_t* dev_status,
                            dspark_stream_t stream);

/*
 * The block sampler's lattice-row branch [G: block-sampler commit - any request that neither
 * walks the lattice greedily nor samples the walk samples the lattice row after the token before,
 * ending the block at a token outside the candidates]. Per request and position j: the whole
 * transformed row s_j (rows and transform as in dspark_topk) with every candidate's entry replaced
 * by its walk value fl32(cand_val[r, j, b] + trans[r, j, prev, b]) (position 0: prev = 0, the row
 * dspark_lattice_score writes from the previous token), sampled as in dspark_sample (temperature,
 * top_p, min_p, U(seed[r], step[r], j, purpose 0), d2t to target ids, q record); prev is the rank
 * of the drawn index among position j's candidates, and a drawn index outside them ends the block.
 * cand_draft [R, B, K] int32 draft indices and cand_val [R, B, K] float32 (from dspark_topk),
 * trans [R, B, K, K] float32 (dspark_lattice_score), all device. Outputs: out_tgt [R, B] and
 * out_idx [R, B] (nullable) int32, -1 after the block's end; n_drafted [R] int32 the block length
 * (1..B); q as in dspark_sample (sparse rows after the end get n = 0). K <= 64.
 * ws: dspark_workspace_size(DSPARK_OP_LATTICE_ROW, R, B, V_d, K).
 */
dspark_status dspark_lattice_row_sample(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                                        int64_t V_d, int64_t ld, const int64_t* row_start,
                                        const int32_t* cand_draft, const float* cand_val,
                                        const float* trans, int32_t K, const int64_t* d2t, int64_t V_t,
                                        float mult, float softcap, float temperature, float top_p,
                                        float min_p, const uint64_t* seed, const uint64_t* step,
                                        int32_t* out_tgt, int32_t* out_idx, int32_t* n_drafted,
                                        const dspark_qrecord* q, void* ws, size_t ws_bytes,
                                        int32_t* dev_status, dspark_stream_t stream);

/*
 * DFlash-2 grouped dynamic convolution over packed block rows.
 * optimum-intel PR #2098 ("Export DFlash v2 and DSpark drafts for PagedAttention and continuous
 * batching"), What does this PR do > DFlash v2: the draft's grouped dynamic convolution shifts its
 * taps along the packed block rows and masks them to the block of the row they produce.
 *   y[i, c] = sum over t < L of k[i, g(c), t] * x[i - t, c], counting a tap only when row i - t
 *             exists and block[i - t] == block[i]; g(c) = c / (C / G).
 * x: [N, C] rows of dtype (row stride ldx >= C), device; k: [N, G, L] float32 taps per produced
 * row and channel group, contiguous, device; block: [N] int32 block of every row, device;
 * y: [N, C] float32 out (row stride ldy >= C), device, caller-owned. Sums are float32 FMAs in tap
 * order. Errors (returned before any launch): DSPARK_EINVAL for a bad dtype or shape, C % G != 0,
 * L outside [1, 16] or a null or misaligned pointer. Nothing is detected on the device, so it
 * takes no status word. Asynchronous on stream.
 */
dspark_status dspark_grouped_conv(const void* x, dspark_dtype dtype, int64_t N, int64_t C, int64_t ldx,
                                  int32_t G, int32_t L, const float* k, const int32_t* block, float* y,
                                  int64_t ldy, dspark_stream_t stream);

/*
 * Failure-detection test hook (not part of the method): sets the poll limit of the first wait
 * for a tile's tensor-core MMAs in dspark_lattice_score, dspark_lattice_chain and
 * dspark_dense_walk, process-wide, for later calls (0xFFFFFFFF restores the default, about 6.7e7
 * polls). A wait that runs out sets DSPARK_ETIMEOUT on *dev_status and the CTA writes no
 * results; it then waits for its MMAs in flight with the full limit before releasing tensor
 * memory, so a limit of 0 makes the timeout path run without leaving work on the GPU.
 */
void dspark_test_set_first_wait_polls(uint32_t polls);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
