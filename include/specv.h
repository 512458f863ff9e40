/*
 * specv.h -- C ABI of libspecv.so: the speculative-decoding verify/accept step
 * with RAPID's inference-time knowledge transfer, on one GB300 (sm_103a).
 *
 * What the step computes (sources, by page title and section):
 *   "RAPID：基于检索增强的推测解码长上下文推理"
 *     - "2) 推理时知识迁移", displayed equation: the enhanced target
 *       p~ = (1 - lambda) * p_t + lambda * p_q  (probability mixture);
 *     - "3) 候选验证机制（伪代码）": softmax of the enhanced target row and
 *       of the draft row, r ~ U(0,1), accept token i iff
 *       r < min(1, p~(x_i) / q(x_i)), otherwise resample and stop.  The
 *       pseudocode mixes logits before the softmax; that reading is the
 *       logit mode, p~ = softmax((1 - lambda) * z_t + lambda * z_q).
 *   "大模型推理的Speculative Decoding原理详解", "数学原理 / 修改的拒绝采样":
 *       the first rejected position ends the step; the rest of the draft is
 *       discarded.
 *   "投机解码（EAGLE）：让小模型猜、大模型验，无损加速 LLM 生成",
 *   "1. 为什么无损": the replacement token is drawn from
 *       normalize(max(0, p~ - q)).
 * Readings where the pages are silent: when all K drafts pass, one bonus
 * token is drawn from p~ at position K+1, which is the target softmax of row
 * K (no draft row exists there); one uniform per sequence serves the
 * resample or the bonus draw; the inverse CDF takes the smallest index whose
 * inclusive prefix sum exceeds u * (total mass); temperature 1, full
 * vocabulary.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers to contiguous row-major memory
 *     owned by the caller; the library never frees or retains them.  The
 *     device memory the library allocates is a scratch workspace for the
 *     row kernels (the streaming kernel's: 16*B*(K+1) bytes of position
 *     statistics, at most 8*B*16*512 bytes of bonus-row segment statistics,
 *     8*B bytes of counters; the other kernels need less or none), plus the
 *     host-buffer calls' staging (see specv_verify_host), one per (device, stream):
 *     created on the first call on that stream that needs it, reused by
 *     every later call on the stream (calls on one stream are ordered, so
 *     they never overlap), kept until the process exits.  A call made while
 *     `stream` is being captured into a CUDA graph uses the stream's existing
 *     workspace (the graph then refers to it: replay such a graph only where
 *     it cannot overlap other calls on that stream); if there is none yet it
 *     takes stream-ordered memory for that call alone (graph-owned).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: they return after the launch;
 *     faults surface at the caller's next synchronisation.
 *   - Host-side argument errors return a status and launch nothing.
 *   - Device-side input errors (a draft token outside [0, V), or lambda
 *     outside [0, 1] or NaN) set out_n_accepted[b] = -1 and fill
 *     out_tokens[b][0..K] with -1.  No trap, no assert.
 *   - A -inf logit masks its entry (probability 0; in the logit mixture a
 *     -inf term of positive weight masks the mixed entry, a term of weight 0
 *     drops out; a drafted token masked in the draft row is accepted iff
 *     p~(x) > 0).  NaN or +inf logits: behaviour unspecified (no fault).
 *   - Uniforms are taken as given; values in [0, 1) give the documented
 *     distribution.
 */
#ifndef SPECV_H
#define SPECV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPECV_F32 = 0,   /* IEEE fp32 logits */
    SPECV_BF16 = 1   /* bfloat16 logits (widened to fp32 exactly on load) */
} specv_dtype;

typedef enum {
    SPECV_PROB_MIX = 0,  /* p~ = (1-l) softmax(z_t) + l softmax(z_q)  (the displayed equation) */
    SPECV_LOGIT_MIX = 1, /* p~ = softmax((1-l) z_t + l z_q)            (the pseudocode) */
    SPECV_GREEDY = 2     /* greedy verification: x_i is accepted iff it is the argmax of
                          * w = z_t + l (z_q - z_t) over row i (w = -inf where z_q = -inf; the
                          * first maximum in index order); the argmax of row n is emitted at
                          * the first mismatch n, the argmax of target row K when every draft
                          * matches.  u_accept and u_resample are not read.  With l = 0 this
                          * is the greedy clause of the EAGLE explainer ("核心思路", step 3):
                          * keep a draft token iff it is the target's most likely token. */
} specv_mode;

typedef enum {
    SPECV_OK = 0,
    SPECV_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, unknown enum */
    SPECV_ERR_UNSUPPORTED = 2,  /* no usable sm_100-family device / launch shape */
    SPECV_ERR_CUDA = 3,         /* a CUDA runtime call failed (see specv_last_cuda_error) */
    SPECV_ERR_NO_MEMORY = 4     /* the scratch workspace could not be allocated */
} specv_status;

/*
 * specv_verify -- one verify/accept step for B sequences of K drafted tokens.
 *
 *   target_logits  [B][K+1][V]  dtype  target scores of the K drafted
 *                                      positions and of position K+1
 *   draft_logits   [B][K][V]    dtype  draft scores of the K drafted positions
 *   draft_tokens   [B][K]       int32  x_i, each in [0, V)
 *   u_accept       [B][K]       fp32   r of the acceptance test, in [0, 1)
 *   u_resample     [B]          fp32   uniform of the resample / bonus draw, in [0, 1)
 *   lambda         [B]          fp32   mixing coefficient per sequence, in [0, 1]
 *   B >= 1, 1 <= K <= 4096, 1 <= V < 2^31, and B*(K+1)*V < 2^62.
 *   out_tokens     [B][K+1]     int32  x_0..x_{n-1}, then the resampled (n < K)
 *                                      or bonus (n = K) token at index n, then -1
 *   out_n_accepted [B]          int32  n = number of accepted drafts (0..K), -1 if invalid
 *
 * Each logit is read from HBM at most once for the statistics; on batches of
 * several waves of CTAs the rows after a sequence's first rejection are not
 * read at all (early exit, specv_plan_flags).  With the resident row kernel
 * and the tile kernels the replacement or bonus token is drawn from the copy
 * of the row held in shared memory; with the sequence-cluster kernel the
 * rejected row pair is read a second time from L2 right after it streamed;
 * with the streaming row kernel the rejected pair is read a second time
 * (from HBM on batches of many waves) and the bonus row only for the one
 * segment its draw lands in.  out_n_accepted[b] = -2 reports an internal
 * copy timeout (a bounded wait that expired; not expected).
 */
specv_status specv_verify(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *lambda, int64_t B, int32_t K,
                          int32_t V, specv_dtype dtype, specv_mode mode, int32_t *out_tokens,
                          int32_t *out_n_accepted, void *stream);

/*
 * specv_verify_host -- specv_verify on inputs and outputs in host memory.
 *
 *   Arguments, layouts and results as specv_verify, except that every array
 *   (the six inputs, out_tokens and out_n_accepted) is a HOST pointer.
 *   chunks         0 = the library's choice (about 64 MiB of logits per
 *                  chunk, at most 16), else 1..64; capped at B.
 *
 * The call copies the inputs into device staging memory that the library
 * owns (one buffer per (device, stream), grown on demand, kept until the
 * process exits), runs the verify step there and copies out_tokens and
 * out_n_accepted back, all asynchronously: the batch is cut into `chunks`
 * runs of whole sequences, each chunk's logits are copied on a copy stream of
 * the library, and each chunk's verify step runs on `stream` as soon as its
 * copy has landed, so the host link and the kernels overlap.  On return
 * nothing has completed yet: the host inputs must stay unchanged, and the
 * outputs unread, until `stream` has completed (cudaStreamSynchronize or an
 * event recorded on it).  The copies are asynchronous only from page-locked
 * host memory; pageable memory gives the same results, with copies that
 * the CUDA runtime may serialise against the host.  Calls on one stream must
 * come from one host thread at a time.
 *
 * The result equals specv_verify's on the same inputs with chunks = 1; with
 * more chunks every sequence is verified by the same kernels on a smaller
 * batch, which may change the launch plan and so the rounding order of the
 * row sums: decisions can then differ only where a uniform lies within
 * rounding error of a decision or CDF boundary.
 *
 * Errors: SPECV_ERR_INVALID_ARG as specv_verify, or chunks outside 0..64;
 * SPECV_ERR_UNSUPPORTED while `stream` is being captured into a CUDA graph
 * (staging may have to grow; capture specv_verify on device buffers
 * instead); SPECV_ERR_NO_MEMORY if the staging memory cannot be allocated.
 */
specv_status specv_verify_host(const void *target_logits, const void *draft_logits,
                               const int32_t *draft_tokens, const float *u_accept,
                               const float *u_resample, const float *lambda, int64_t B, int32_t K,
                               int32_t V, specv_dtype dtype, specv_mode mode, int32_t *out_tokens,
                               int32_t *out_n_accepted, int32_t chunks, void *stream);

/*
 * specv_verify_host_direct -- specv_verify on inputs and outputs in host
 * memory that the device reads and writes in place: the kernels load the rows
 * they reach straight over the host link, so only those rows cross it (the
 * pages' loop stops at the first rejection -- RAPID explainer, "3) 候选验证机制
 * （伪代码）" -- and on batches of several waves positions after a published
 * rejection read nothing), with no staging copy to wait for.
 *
 *   Arguments, layouts and results as specv_verify_host, without `chunks`.
 *   Every buffer must be device-accessible: page-locked and mapped
 *   (cudaHostAlloc, cudaHostRegister, or PyTorch's pin_memory), or ordinary
 *   host memory on a device that reads pageable memory
 *   (cudaDevAttrPageableMemoryAccess); device memory is accepted as well.
 *
 * Asynchronous on `stream` like specv_verify: the outputs are complete once the
 * stream has completed.  The kernels that stage rows with bulk copies are not
 * planned here (the register-load kernels read host memory the same way as
 * device memory); results equal specv_verify's on the same plan.  Errors as
 * specv_verify, and SPECV_ERR_UNSUPPORTED when a buffer is not
 * device-accessible (nothing is launched).
 */
specv_status specv_verify_host_direct(const void *target_logits, const void *draft_logits,
                                      const int32_t *draft_tokens, const float *u_accept,
                                      const float *u_resample, const float *lambda, int64_t B,
                                      int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                      int32_t *out_tokens, int32_t *out_n_accepted,
                                      void *stream);

/*
 * specv_verify_host_early_exit -- specv_verify_host that copies only the rows
 * the verify step reaches.  The pages' loop stops at the first rejection
 * (RAPID explainer, "3) 候选验证机制（伪代码）"; SD explainer, "修改的拒绝采样":
 * the rest of the draft is discarded), so a sequence's rows after its first
 * rejected position never influence its outputs.  The call copies the batch
 * position by position: level i sends row pair (b, i) (level K: target row
 * K) of every sequence still live over the host link, decides position i of
 * those sequences on the device, reads the B live flags back (one small copy
 * and a wait on `stream` per level), and stops copying a sequence once a
 * position clearly rejects (a margin of 1e-4 relative keeps every row the
 * verify step could read under other rounding).  The ordinary verify step then
 * runs on the staged batch.
 *
 *   Arguments, layouts and results as specv_verify_host (HOST pointers; the
 *   outputs equal specv_verify's with a one-chunk plan), without `chunks`;
 *   out_h2d_bytes and out_d2h_bytes (each may be NULL) receive the bytes
 *   copied to the device and read back (the outputs and the live flags).
 *
 * Blocking: the call returns once every row it sends has been copied (it
 * waits on `stream` after each level); the final verify step and the two
 * output copies are still in flight on `stream` at return.  Staging memory is
 * shared with specv_verify_host (per device and stream).  Errors as
 * specv_verify_host (SPECV_ERR_UNSUPPORTED under stream capture).
 */
specv_status specv_verify_host_early_exit(const void *target_logits, const void *draft_logits,
                                          const int32_t *draft_tokens, const float *u_accept,
                                          const float *u_resample, const float *lambda,
                                          int64_t B, int32_t K, int32_t V, specv_dtype dtype,
                                          specv_mode mode, int32_t *out_tokens,
                                          int32_t *out_n_accepted, int64_t *out_h2d_bytes,
                                          int64_t *out_d2h_bytes, void *stream);

/*
 * specv_shard_bounds -- the sequences [*lo, *hi) of shard `shard` when a batch
 * of B sequences is split over n_shards (1..64) shards for
 * specv_verify_sharded_host: contiguous runs in order, lo = shard * (B /
 * n_shards) + min(shard, B mod n_shards), sizes differing by at most one (a
 * shard is empty when B < n_shards).  Sequences are independent (SD
 * explainer, "批量投机（Batched Speculation）": each sequence of a batch is
 * verified on its own), so the shards' outputs concatenate to the batch's.
 * Host-only arithmetic.  SPECV_ERR_INVALID_ARG for a NULL output, B < 0 or a
 * shard index outside [0, n_shards).
 */
specv_status specv_shard_bounds(int64_t B, int32_t n_shards, int32_t shard, int64_t *lo,
                                int64_t *hi);

/*
 * specv_verify_sharded_host -- one batch in host memory verified on several
 * devices: shard g (specv_shard_bounds) runs specv_verify_host on device
 * devices[g] (a device may appear more than once: its shards then run on
 * separate streams of that device), and its out_tokens / out_n_accepted rows
 * land at the shard's offset in the caller's host arrays.  Arguments and
 * layouts as specv_verify_host, all arrays HOST pointers (page-locked memory
 * lets the shards' copies run at the same time); devices [n_shards], n_shards
 * in 1..64.  No data crosses devices: no collective, no peer memory.
 *
 * Unlike specv_verify_host the call is synchronous: it returns after every
 * shard has completed, the outputs in place.  It uses streams and staging
 * memory the library owns per (device, shard index), and leaves the calling
 * thread's current device unchanged.  Each sequence's outputs equal those of
 * specv_verify_host on the whole batch whenever the launch plan is the same
 * (it depends on a shard's size); otherwise decisions can differ only within
 * rounding of a decision or CDF boundary (greedy verification not at all
 * outside its tie band).
 *
 * Errors: SPECV_ERR_INVALID_ARG as specv_verify_host, for a NULL `devices`,
 * n_shards outside 1..64, or a device index that does not exist; the first
 * shard's error otherwise (shards already launched are waited for).
 */
specv_status specv_verify_sharded_host(const void *target_logits, const void *draft_logits,
                                       const int32_t *draft_tokens, const float *u_accept,
                                       const float *u_resample, const float *lambda, int64_t B,
                                       int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                       int32_t *out_tokens, int32_t *out_n_accepted,
                                       int32_t n_shards, const int32_t *devices);

/*
 * specv_verify_debug -- specv_verify plus the intermediate probabilities, for
 * tests.  Same kernels and the same arithmetic as specv_verify; the extra
 * outputs (device pointers, each may be NULL) are:
 *   out_ptilde_at_x [B][K]     fp32  p~(x_i) as the kernel computed it
 *   out_q_at_x      [B][K]     fp32  q(x_i)
 *   out_lse         [B][K+1][2] fp32 natural-log normalisers: [.][i][0] of the
 *                                     p~ source row (target row in probability
 *                                     mode and at i = K, mixed row in logit
 *                                     mode), [.][i][1] of the draft row
 *                                     (undefined at i = K)
 * For a given input, out_tokens and out_n_accepted equal specv_verify's.
 * SPECV_GREEDY computes no probabilities: it returns SPECV_ERR_UNSUPPORTED.
 */
specv_status specv_verify_debug(const void *target_logits, const void *draft_logits,
                                const int32_t *draft_tokens, const float *u_accept,
                                const float *u_resample, const float *lambda, int64_t B,
                                int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                int32_t *out_tokens, int32_t *out_n_accepted,
                                float *out_ptilde_at_x, float *out_q_at_x, float *out_lse,
                                void *stream);

/*
 * specv_plan -- host-only query of the launch specv_verify would make for
 * these sizes (no device work, no allocation).  Outputs may be NULL:
 *   kernel:  0 = small-vocabulary tile kernel, 1 = streaming cluster row
 *            kernel, 2 = resident cluster row kernel (slices staged in shared
 *            memory by TMA; chosen when rows start on 16-byte boundaries and
 *            a slice fits shared memory, and the grid is a single wave),
 *            3 = small-vocabulary tile kernel with TMA-staged, double-buffered
 *            tiles (16-byte aligned rows), 4 = sequence-cluster row kernel (one
 *            cluster of 16 CTAs per sequence streams every position, decides
 *            it and draws its token in one launch with no workspace; sampling
 *            rules, device memory, grids of one wave of 2 to 4 CTAs per SM).
 *            For tests, the environment variable SPECV_ROWS_VARIANT=stream or
 *            =resident forces kernel 1 or 2, and SPECV_CLUSTER_SIZE=1..16
 *            forces the cluster size of the row kernels (either one, or
 *            SPECV_SAMPLE_SPLIT, rules out kernel 4).
 *   cluster: CTAs per thread-block cluster splitting each row (1 for kernel 0)
 *   ctas:    CTAs launched by a row kernel; tiles of sequences for kernels 0, 3
 *   workspace_bytes: scratch bytes of the row kernels' workspace (kept per
 *            device and stream, see specv_verify)
 * Returns SPECV_ERR_INVALID_ARG for sizes specv_verify would reject.
 */
specv_status specv_plan(int64_t B, int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                        int32_t *kernel, int32_t *cluster, int64_t *ctas,
                        int64_t *workspace_bytes);

/*
 * specv_plan_flags -- host-only query of how the launch specv_verify would
 * make for these sizes behaves (no device work, no allocation).  *flags
 * (not NULL) receives a bit set:
 *   SPECV_PLAN_EARLY_EXIT  -- the streaming row kernel runs position-major and
 *       a position whose sequence already has a published rejection at an
 *       earlier position reads none of its rows (the pages' loop stops at the
 *       first rejection: RAPID explainer, "3) 候选验证机制（伪代码）"; SD
 *       explainer, "修改的拒绝采样").  Taken on grids of more than two waves of
 *       CTAs; the environment variable SPECV_EARLY_EXIT=0 turns it off.  The
 *       outputs do not depend on it.
 *   SPECV_PLAN_SPLIT_DRAWS -- the token draws run as a second launch
 *       (grids of one or two waves; SPECV_SAMPLE_SPLIT=0/1 forces either way).
 * Returns SPECV_ERR_INVALID_ARG for sizes specv_verify would reject.
 */
#define SPECV_PLAN_EARLY_EXIT 1u
#define SPECV_PLAN_SPLIT_DRAWS 2u
specv_status specv_plan_flags(int64_t B, int32_t K, int32_t V, specv_dtype dtype,
                              specv_mode mode, uint32_t *flags);

/*
 * specv_verify_tree -- the verify/accept step for a tree of drafted tokens per
 * sequence (the speculative-decoding explainer's "Tree Speculation": several
 * candidate branches per position verified at once, so that another branch can
 * be accepted when one is rejected).  Rule (a reading; the pages give none for
 * several branches): node 0 is the root; the children of node u were drawn
 * independently from the draft distribution q_u; starting at the root with
 * p = p~_u, u's children are tested in index order, x_c accepted iff
 * u_accept[c] < min(1, p(x_c)/q_u(x_c)); a rejection replaces p by
 * normalize(max(0, p - q_u)); an acceptance moves on to c.  When every child is
 * rejected the token is drawn from p (inverse CDF with u_resample[b]); at a
 * node without children, the bonus token from p~_u.  p~_u mixes the target row
 * of u with q_u by `mode`, or is the target softmax when u has no draft row.
 * A chain (parent[j] = j - 1) is specv_verify.
 *   target_logits [B][N+1][V]  target row of every node (row 0: the root)
 *   draft_logits  [B][M][V]    draft rows (may be NULL when M == 0)
 *   parent        [B][N+1]     int32: -1 at node 0, parent[j] in [0, j) else
 *   draft_row     [B][N+1]     int32: the draft row (in [0, M)) u's children
 *                              were drawn from, -1 for a node without children
 *   tokens        [B][N+1]     int32: token of node j (entry 0 unused)
 *   u_accept      [B][N+1]     fp32: uniform of node j's test (entry 0 unused)
 *   u_resample [B], lambda [B] fp32
 *   mode          SPECV_PROB_MIX or SPECV_LOGIT_MIX
 *   out_tokens    [B][N+1]     accepted tokens along the path, then the drawn
 *                              token, then -1
 *   out_path      [B][N+1]     the accepted nodes in order, then -1
 *   out_n         [B]          number of accepted nodes; -1 for an invalid
 *                              sequence (bad parent, draft_row or token, a node
 *                              with children but no draft row, lambda outside
 *                              [0, 1]): then every output entry is -1
 * Every node's rows are read once for their statistics; the walk reads the
 * rows of the nodes it visits again (one pass per rejection, one for the final
 * draw).  Scratch as specv_verify's streaming kernel (16 bytes per node + one
 * counter per sequence).  Host argument errors (null pointers, B < 1, N < 0 or
 * > 4096, M < 0, V < 1, overflowing sizes, unknown enums) return
 * SPECV_ERR_INVALID_ARG and launch nothing.
 */
specv_status specv_verify_tree(const void *target_logits, const void *draft_logits,
                               const int32_t *parent, const int32_t *draft_row,
                               const int32_t *tokens, const float *u_accept,
                               const float *u_resample, const float *lambda, int64_t B, int32_t N,
                               int32_t M, int32_t V, specv_dtype dtype, specv_mode mode,
                               int32_t *out_tokens, int32_t *out_path, int32_t *out_n,
                               void *stream);

/*
 * specv_acceptance_rates -- the exact acceptance probability of every drafted
 * position, for host policies such as specv_choose_k.  A draft token x ~ q is
 * accepted with probability min(1, p~(x)/q(x)) (the RAPID explainer's
 * "3) 候选验证机制" loop), so position i of sequence b is accepted with
 *   alpha[b][i] = sum_v min(p~_v, q_v)  (1 minus the total variation distance),
 * the per-position rate on which the speculative-decoding explainer builds
 * its expected-token count ("加速效果分析").
 *   target_logits [B][K+1][V], draft_logits [B][K][V], lambda [B]: as for
 *   specv_verify (rows K of the target are not read); mode PROB_MIX or
 *   LOGIT_MIX (SPECV_GREEDY: SPECV_ERR_UNSUPPORTED);
 *   out_alpha [B][K] fp32, device; NaN where lambda is outside [0, 1].
 * Two passes over every drafted row pair (statistics, then the overlap sum),
 * the second mostly from L2; no scratch, no allocation; asynchronous on
 * `stream`.  Host argument errors as for specv_verify.
 */
specv_status specv_acceptance_rates(const void *target_logits, const void *draft_logits,
                                    const float *lambda, int64_t B, int32_t K, int32_t V,
                                    specv_dtype dtype, specv_mode mode, float *out_alpha,
                                    void *stream);

/*
 * specv_choose_k -- host-only draft-length policy (no device work): the K in
 * [k_min, k_max] that maximises the expected tokens of one step per unit of
 * step cost,
 *   tokens(K) = 1 + alpha + ... + alpha^K   (accepted prefix + the final token,
 *                                             positions accepted independently
 *                                             with probability alpha),
 *   cost(K)   = cost_verify_fixed + K * (cost_draft + cost_verify_per_token),
 * the smallest such K on ties.  This is the adaptive draft length of the EAGLE
 * explainer ("4. 草稿长度和接受率的权衡": lengthen the draft when recent
 * acceptance is high, shorten it when low) made concrete with the expected
 * token count of the speculative-decoding explainer ("加速效果分析").
 * alpha would typically be a running mean of specv_acceptance_rates.
 * Returns -1 for alpha outside [0, 1] or NaN, k_min < 1, k_max < k_min or
 * > 4096, a negative cost, or a step cost of zero.
 */
int32_t specv_choose_k(double alpha, double cost_draft, double cost_verify_fixed,
                       double cost_verify_per_token, int32_t k_min, int32_t k_max);

/*
 * specv_verify_noalloc -- specv_verify for callers that cannot let a library
 * allocate device memory while they run: an engine that hands all of HBM to
 * its own pools up front, a decode loop where an allocation could stall or
 * fail, or code that must never see an out-of-memory error from this call.
 * (The pages have no counterpart: this is an interface choice of this
 * library, not part of the method.)
 *
 * Same arguments, semantics and outputs as specv_verify; it always runs the
 * streaming cluster row kernel, whose scratch (position statistics and
 * per-sequence counters) lives in a fixed 1 MiB array inside the library's
 * device image instead of memory allocated per call.  Limits and rules:
 *   - B * (K+1) <= 49152 and B <= 65536; larger calls return
 *     SPECV_ERR_INVALID_ARG and launch nothing;
 *   - the array exists once per GPU and is shared by every call on that GPU:
 *     calls whose work overlaps on the GPU (other streams, other host
 *     threads) race on it; serialise them (e.g. use one stream);
 *   - the first call on a device looks up the array's address (this also
 *     loads the library's device code there): make it before any CUDA graph
 *     capture;
 *   - no cudaMalloc/cudaFree or other allocating call is made (the counters
 *     are cleared with cudaMemsetAsync on `stream`).
 */
specv_status specv_verify_noalloc(const void *target_logits, const void *draft_logits,
                                  const int32_t *draft_tokens, const float *u_accept,
                                  const float *u_resample, const float *lambda, int64_t B,
                                  int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                  int32_t *out_tokens, int32_t *out_n_accepted, void *stream);

/* Human-readable name of a status. Never NULL. */
const char *specv_status_string(specv_status status);

/*
 * specv_release_stream -- frees what the library keeps for (current device,
 * stream): the row kernels' scratch (including buffers it outgrew) and the
 * host-buffer calls' staging memory, copy stream and events.  It waits for
 * the stream's queued work first.  Call it before destroying a stream on
 * which the library ran, once no CUDA graph captured from library calls on
 * that stream will be replayed (a graph refers to the scratch by address).
 * The next call on the stream allocates afresh.  SPECV_ERR_UNSUPPORTED while
 * the stream is being captured; SPECV_ERR_CUDA if waiting fails.
 */
specv_status specv_release_stream(void *stream);

/* Text of the CUDA error behind the most recent SPECV_ERR_CUDA on this
 * thread ("" if none).  Never NULL. */
const char *specv_last_cuda_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int32_t specv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECV_H */
