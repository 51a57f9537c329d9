/*
 * spv.h -- speculative-sampling verify step on one GB300 (sm_103a).
 *
 * C ABI of libspv.so.  All tensors are caller-owned DEVICE memory; the
 * library allocates nothing and frees nothing.  Every compute call is
 * asynchronous on the caller's CUDA stream (a cudaStream_t passed as void*;
 * NULL = legacy default stream) and returns after the launch.  Argument
 * errors are found on the host before anything is launched.
 *
 * Sources (web pages; section names are the pages' own):
 *   [SD]  "Speculative Decoding: How Draft-Model Parallelism Cuts LLM
 *         Inference Latency", section "The four-phase loop" steps 2-4 and
 *         "The acceptance criterion and why it is exact".
 *   [SPD] "Speculative Pipeline Decoding: Higher-Accuracy Drafting with
 *         Hidden Latency via Pipeline Parallelism", streaming verification
 *         (one in-flight token per cycle: gamma = 1; greedy = exact argmax
 *         match; sampling = standard rejection sampling).
 *   [SSD] "Speculative Speculative Decoding" (review of arXiv 2603.03251),
 *         Figure 2 and "Core Technical Barrier": geometric fan-out
 *         F_k = F_0 * a_p^(k/(1+r)) of bonus-token candidates taken from the
 *         top ranks of the draft logits, excluding the sampled token.
 *
 * Layouts are row-major with the vocabulary axis V contiguous.  A "row" is
 * one V-vector of logits.  Logits are fp32 or bf16 (spv_dtype).
 */
#ifndef SPV_H
#define SPV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPV_OK = 0,
    SPV_ERR_INVALID_ARG = 1, /* bad pointer, size, dtype, temperature, workspace */
    SPV_ERR_CUDA = 2,        /* a CUDA runtime call or launch failed */
    SPV_ERR_UNSUPPORTED = 3, /* valid request outside what the build supports */
    SPV_ERR_BAD_ROW = 4,     /* per-sequence: NaN/+inf logits, an all -inf row,
                                or a draft token outside [0, V) */
    SPV_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (workspace word) */
} spv_status;

typedef enum { SPV_F32 = 0, SPV_BF16 = 1 } spv_dtype;

/* Limits of the library. */
#define SPV_MAX_GAMMA 32     /* draft tokens per sequence */
#define SPV_MAX_FANOUT 64    /* F_k per position */
#define SPV_MAX_FANOUT_ROWS 64 /* K + 1 positions in the fan-out */
#define SPV_SAMPLER_BLOCK 1024 /* ids per sampler block (part of the sampling rule) */
#define SPV_SAMPLER_SUB 32     /* ids per sampler sub-block (part of the sampling rule) */
#define SPV_MAX_TRIALS 64    /* residual rejection trials before the direct draw */
#define SPV_MAX_TOP_K 64     /* top_k of spv_verify_chain_filtered */
#define SPV_MAX_TREE_NODES 64 /* nodes of a spv_verify_tree draft tree (root included) */

/*
 * spv_verify_chain -- [SD] steps 3 and 4 for B independent sequences.
 *
 * For each sequence b and draft position i = 0..gamma-1:
 *   p_i = softmax(target[b,i,:] / T), q_i = softmax(draft[b,i,:] / T);
 *   x_i = draft_tokens[b,i] is accepted iff p_i(x_i) > 0 and
 *   r[b,i] * q_i(x_i) <= p_i(x_i)   ([SD] step 3's ratio test without a division).
 * k = number of leading accepted tokens (stop at the first rejection).
 * Emitted: x_0..x_{k-1}, then one more token:
 *   k <  gamma: a draw from norm(max(0, p_k - q_k))   (residual, [SD] step 4)
 *   k == gamma: a draw from p_gamma                   (bonus, [SD] step 4)
 * T == 0 selects greedy semantics ([SPD]): identical to spv_verify_greedy;
 * draft_logits, r and sample_keys are then not read and may be NULL.
 *
 * Sampling rule (exact for the stated distributions; both the library and
 * any independent checker follow it): ids are grouped in blocks of
 * SPV_SAMPLER_BLOCK ids and each block in sub-blocks of SPV_SAMPLER_SUB ids.
 * A draw from a distribution P is an exponential race at three levels: the
 * block with the smallest E / P(block) wins, then inside it the sub-block
 * with the smallest E / P(sub-block), then the id with the smallest E / P(id)
 * (E = -ln U, ties to the lower index).  The residual is drawn by up to
 * SPV_MAX_TRIALS rejection trials (draw x from p_k, accept iff
 * q_k(x) <= (1 - v) p_k(x)), then, if none is accepted, by the same race over
 * max(0, p_k - q_k) directly.  U = ((w >> 8) + 1) * 2^-24 for one 32-bit
 * word w of Philox4x32-10 with key (low, high half of sample_keys[b]) and
 * counter (n / 4, stream, trial, 0), word n % 4, where n is the block index,
 * the sub-block's index within its block (0..31) or the id's offset within
 * its sub-block (0..31); streams 1 / 2 / 3 block / sub-block / id race, 4
 * trial acceptance (n = 0), 5 / 6 / 7 the direct residual race.  Trials are
 * numbered from 0; the bonus is trial 0.  The position of the draw is not in
 * the counter: a sequence makes exactly one draw, so its variates are i.i.d.
 * whatever the position, and given the winning block (sub-block) the
 * sub-block (id) variates are fresh -- every level of the race stays exact.
 *
 * Arguments (all device pointers unless noted):
 *   target_logits  [B, gamma+1, V] dtype
 *   draft_logits   [B, gamma, V]   dtype            (T > 0)
 *   draft_tokens   [B, gamma] int32
 *   r              [B, gamma] fp32, values in (0, 1] (T > 0)
 *   sample_keys    [B] uint64, one key per sequence (T > 0)
 *   B >= 1, 1 <= gamma <= SPV_MAX_GAMMA, V >= 2, temperature >= 0 finite.
 *   accept_count   [B] int32 out: k, or -1 for a bad row
 *   out_tokens     [B, gamma+1] int32 out: k+1 ids, then -1
 *   out_pq         [B, gamma, 2] fp32 out, optional: p_i(x_i), q_i(x_i)
 *   out_resid_norm [B] fp32 out, optional: sum_x max(0, p_k - q_k) when
 *                  k < gamma, 1 for the bonus.  Costs one extra read of the
 *                  rejected row pair per sequence; pass NULL on the hot path.
 *   row_status     [B] int32 out, optional: SPV_OK, SPV_ERR_BAD_ROW, or
 *                  SPV_ERR_TIMEOUT when the workspace's error word records a
 *                  bounded wait that gave up (the sequence's statistics may be
 *                  incomplete; its accept_count and out_tokens are then -1)
 *   workspace      device scratch of >= spv_chain_workspace_bytes(B,gamma,V)
 *                  bytes, 256-byte aligned.  Its first 4 bytes are a sticky
 *                  error word (see spv_workspace_status); bytes 8..15 are
 *                  the counter through which the streaming pass hands out
 *                  work items, which every call leaves at zero.  Zero-fill
 *                  the workspace once before its first use, and again after
 *                  a call that returned an error (its kernels may not all
 *                  have run).  One workspace must not be shared by calls
 *                  that may overlap on the GPU.
 *   stream         cudaStream_t (void*).  Two kernels are enqueued: the
 *                  streaming pass and, as a programmatic dependent launch,
 *                  the per-sequence finalize.
 * Bad rows do not stop the launch: their outputs are -1 and row_status is
 * SPV_ERR_BAD_ROW.  Returns SPV_OK once the work is enqueued.
 */
spv_status spv_verify_chain(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                            const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                            int B, int gamma, int V, float temperature,
                            int32_t *accept_count, int32_t *out_tokens, float *out_pq,
                            float *out_resid_norm, int32_t *row_status,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes spv_verify_chain needs (also valid for T == 0). */
size_t spv_chain_workspace_bytes(int B, int gamma, int V);

/*
 * spv_verify_chain_saguaro -- spv_verify_chain_cached for drafts drawn by
 * Saguaro sampling ([SSD] "Key Innovations" / Table 7b, logit bonus C,
 * Theorem 15: the cache hit rate grows with C; C = 1 is plain sampling).
 * Reading: at draft position i the draft drew x_i from
 *   q_C,i(x) = q_i(x) w_i(x) / sum_y q_i(y) w_i(y),  w_i(x) = 1/C if x is one
 * of position i's cached candidates (cache_ids entries off_i .. off_i + F_i
 * - 1, ids outside [0, V) ignored, repeats counted once), else 1.
 * The verify step runs on (p_i, q_C,i) -- [SD] steps 3 and 4 with q_C as the
 * draft distribution, so the emitted tokens stay distributed as p -- and the
 * outcome is looked up in the cache as by spv_verify_chain_cached.  out_pq
 * holds p_i(x_i), q_C,i(x_i); out_resid_norm sum max(0, p_k - q_C,k).
 *   C           > 0, finite (C > 1 moves residual mass onto the cached ids)
 *   V           <= 1,048,576 (else SPV_ERR_UNSUPPORTED)
 * Other arguments, the workspace and T == 0 (greedy; C plays no part) as
 * spv_verify_chain_cached.
 */
spv_status spv_verify_chain_saguaro(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                    const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                                    int B, int gamma, int V, float temperature,
                                    const int32_t *cache_ids, const int32_t *fanout, float C,
                                    int32_t *accept_count, int32_t *out_tokens, float *out_pq,
                                    float *out_resid_norm, int32_t *row_status, int32_t *cache_slot,
                                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * spv_verify_chain_cached -- spv_verify_chain followed, in the same kernels,
 * by the speculation-cache lookup of [SSD] Algorithm 1 (the speculator's
 * test whether the verify outcome is in its cache) with the cache of
 * Figure 2: for each position k = 0..gamma, F_k candidate tokens.
 *
 * The outcome of sequence b is (k, t*): k = accept_count[b] and t* =
 * out_tokens[b, k], the residual draw (k < gamma) or the bonus (k = gamma).
 * The cache entries of sequence b are cache_ids[b, :], k-major: entries
 * off_k .. off_k + F_k - 1 (off_k = F_0 + ... + F_{k-1}) are the candidates
 * for position k -- exactly the layout spv_fanout_topk writes for the draft
 * rows of positions 0..gamma with K = gamma.  The outcome hits when one of
 * position k's entries equals t*; cache_slot[b] is then that entry's index
 * in 0 .. sum_k F_k - 1 (the lowest one if the list repeats an id), else -1.
 * A bad row never hits (cache_slot -1).
 *
 *   cache_ids   [B, sum_k F_k] int32 (device), any values (-1 never matches
 *               an emitted token)
 *   fanout      gamma + 1 ints, HOST array, 0 <= F_k <= SPV_MAX_FANOUT
 *   cache_slot  [B] int32 out (device)
 * All other arguments, the workspace and the T == 0 (greedy) semantics are
 * those of spv_verify_chain.  A null cache_ids, fanout or cache_slot, or an
 * F_k out of range, returns SPV_ERR_INVALID_ARG before any launch.
 */
spv_status spv_verify_chain_cached(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                   const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                                   int B, int gamma, int V, float temperature,
                                   int32_t *accept_count, int32_t *out_tokens, float *out_pq,
                                   float *out_resid_norm, int32_t *row_status,
                                   const int32_t *cache_ids, const int32_t *fanout, int32_t *cache_slot,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * spv_verify_chain_filtered -- spv_verify_chain on top-k / top-p filtered
 * distributions ([SPD] "Evaluation": the sampled runs use top-k = 50 and
 * top-p = 1.0 at T = 1).  Each target row i = 0..gamma and draft row
 * i = 0..gamma-1 is filtered the same way:
 *   1. keep the top_k ids by logit (descending, -0.0 equal to +0.0, ties to
 *      the lower id);
 *   2. p'(x) = exp((z_x - z_max) / T) / sum over the kept ids;
 *   3. if top_p < 1, keep only the shortest prefix of them (in that order)
 *      whose p' sum reaches top_p, and renormalise over it.
 * Every other id has probability 0.  [SD] steps 3 and 4 then run on p', q':
 * x_i stands iff p'_i(x_i) > 0 and r_i q'_i(x_i) <= p'_i(x_i); at the first
 * rejection k one token is drawn from norm(max(0, p'_k - q'_k)), else the
 * bonus from p'_gamma.  The draw is an exponential race over the kept ids
 * of target row k: the id x with the smallest E_x / w(x) wins (w the
 * residual or bonus mass, E_x = -ln U with U from Philox4x32-10 as for
 * spv_verify_chain, counter (x / 4, 8, 0, 0), word x % 4; ties to the lower
 * id).  A rejection whose residual has no mass (a draft token outside q's
 * support with p' = q' elsewhere) makes the row bad.
 *
 *   top_k       1 .. SPV_MAX_TOP_K (top_k >= V keeps every id)
 *   top_p       in (0, 1]; 1 disables the nucleus cut
 *   out_pq      p'_i(x_i), q'_i(x_i); out_resid_norm: sum max(0, p'_k - q'_k)
 *               (k < gamma) or 1 (bonus) -- free here, no extra read
 *   workspace   >= spv_filtered_workspace_bytes(B, gamma, V) bytes, 256-byte
 *               aligned, zero-filled once (first 4 bytes: error word)
 * T == 0 selects the greedy rule of spv_verify_greedy (no top-k filter
 * changes an argmax).  Other arguments as spv_verify_chain.
 */
spv_status spv_verify_chain_filtered(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                     const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                                     int B, int gamma, int V, float temperature, int top_k, float top_p,
                                     int32_t *accept_count, int32_t *out_tokens, float *out_pq,
                                     float *out_resid_norm, int32_t *row_status,
                                     void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes spv_verify_chain_filtered needs (also valid for T == 0). */
size_t spv_filtered_workspace_bytes(int B, int gamma, int V);

/*
 * spv_verify_tree -- verify of a draft token tree per sequence.  The pages
 * name draft trees ([SPD] tree drafting of width 4; tree verification with
 * k = 21 nodes in the benchmark study) but give no verification rule; this
 * follows the published multi-round speculative sampling for token trees
 * (SpecInfer), which keeps the emitted tokens distributed as the target's.
 * Node 0 is the root (the context); node v >= 1 holds token tokens[b,v] and
 * hangs from parent[b,v] < v.  target row v is p at node v (the next-token
 * distribution after the path to v), draft row v is q at node v, from which
 * v's children were drawn i.i.d.  From the root: the children c of node u
 * are tested in index order against
 *   P_m = max(0, p_u - s_m q_u) / N_m,  s_0 = 0, N_0 = 1, s_{m+1} = s_m + N_m,
 *   N_m = sum_x max(0, p_u(x) - s_m q_u(x)),
 * m = children rejected so far: c (token x) is accepted iff P_m(x) > 0 and
 * r[b,c] q_u(x) <= P_m(x), and the walk descends into it.  When every child
 * of u is rejected one token is drawn from P_m (the chain's rejection trials
 * from p_u with q scaled by s_m, then the direct residual race); at a leaf
 * the bonus token from p_u.  Draws follow spv_verify_chain's sampling rule
 * (one draw per sequence).  A tree that is one path is
 * spv_verify_chain exactly (r[b, i+1] <-> r[b, i]).  T == 0: descend into the
 * first child whose token is the argmax of p_u (lowest id on ties), emit the
 * last node's argmax; draft_logits, r and sample_keys are then not read.
 *   target_logits, draft_logits  [B, N, V] dtype (device)
 *   parent, tokens               [B, N] int32 (device); parent[b,0] = -1
 *   r                            [B, N] fp32 in (0, 1] (r[b,0] unused)
 *   1 <= N <= SPV_MAX_TREE_NODES
 *   accept_count [B] out: accepted nodes k (-1 for a bad row)
 *   out_tokens   [B, N] out: the k accepted tokens, the drawn one, then -1
 *   out_nodes    [B, N] out, optional: the k accepted nodes, then -1
 *   row_status   [B] out, optional
 *   workspace    >= spv_tree_workspace_bytes(B, N, V) bytes (zero-filled once)
 * Bad rows: a parent outside [0, v) or a token outside [0, V); NaN / +inf or
 * no finite logit in any target row, or in the draft row of a node with
 * children; a rejection whose residual has no mass.
 */
spv_status spv_verify_tree(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                           const int32_t *parent, const int32_t *tokens, const float *r,
                           const uint64_t *sample_keys, int B, int N, int V, float temperature,
                           int32_t *accept_count, int32_t *out_tokens, int32_t *out_nodes, int32_t *row_status,
                           void *workspace, size_t workspace_bytes, void *stream);

size_t spv_tree_workspace_bytes(int B, int N, int V);

/* Bytes of device memory behind spv_verify_chain_noalloc (per GPU, held from
 * library load until process exit). */
#define SPV_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)

/*
 * spv_verify_chain_noalloc -- spv_verify_chain for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an
 * interface addition, not part of the method.
 *
 * Who needs it: a caller that cannot hand the library a workspace -- a
 * serving loop whose device memory is entirely pre-reserved by its own pool,
 * a host program that links this library but manages no device memory, or
 * code running where cudaMalloc is not allowed or would stall the device
 * (cudaMalloc / cudaFree may synchronise).  Same arguments, semantics and
 * kernels as spv_verify_chain, without workspace / workspace_bytes: the
 * scratch space is a fixed array of SPV_NOALLOC_SCRATCH_BYTES in the
 * library's own device memory.  The call allocates and frees nothing.
 *
 *   - Returns SPV_ERR_UNSUPPORTED when the call needs more scratch than the
 *     array holds: spv_chain_workspace_bytes(B, gamma, V) >
 *     SPV_NOALLOC_SCRATCH_BYTES for T > 0, spv_greedy_workspace_bytes(B,
 *     gamma, V) > SPV_NOALLOC_SCRATCH_BYTES for T == 0 (e.g. B = 64,
 *     gamma = 4, V = 151,936 needs about 0.7 MB at T > 0, B = 256 about
 *     2.9 MB).  Other argument errors are those of spv_verify_chain.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make
 *     that first call before any stream capture.
 *   - Every call on a device uses the same array, and the array keeps the
 *     last call's contents.  Calls whose kernels may overlap on the GPU (on
 *     different streams, or from different host threads) race on it and
 *     must be serialised by the caller.  Each call first clears the array's
 *     16-byte call header -- the error word, the self-test flag and the
 *     streaming pass's work-item counter -- with an asynchronous memset on
 *     `stream`, so a call that failed part-way (the caller cannot zero-fill
 *     this array) leaves nothing that changes the next call's results.
 *   - A bounded wait of the call's streaming pass that gave up cannot be read
 *     back with spv_workspace_status (the caller has no pointer to the
 *     array); the call reports it in its outputs instead: accept_count -1,
 *     out_tokens -1 and row_status SPV_ERR_TIMEOUT for every sequence.
 */
spv_status spv_verify_chain_noalloc(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                    const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                                    int B, int gamma, int V, float temperature,
                                    int32_t *accept_count, int32_t *out_tokens, float *out_pq,
                                    float *out_resid_norm, int32_t *row_status, void *stream);

/*
 * spv_verify_greedy -- T = 0 ([SPD] streaming verification: a draft token
 * stands only if it is the target's most likely token).  a_i = argmax_x target[b,i,x] (lowest id on ties,
 * -0.0 equal to +0.0); x_i accepted iff x_i == a_i; stop at the first
 * mismatch k and emit a_k there (a_gamma when all matched).  Draft logits are
 * not needed.  Arguments as in spv_verify_chain; workspace of
 * >= spv_greedy_workspace_bytes(B, gamma, V) bytes (zero-filled once).
 */
spv_status spv_verify_greedy(const void *target_logits, spv_dtype dtype, const int32_t *draft_tokens,
                             int B, int gamma, int V,
                             int32_t *accept_count, int32_t *out_tokens, int32_t *row_status,
                             void *workspace, size_t workspace_bytes, void *stream);

size_t spv_greedy_workspace_bytes(int B, int gamma, int V);

/*
 * spv_fanout_topk -- [SSD] Figure 2: for each sequence b and position
 * k = 0..K, the F_k ids with the largest draft logit draft[b,k,:], skipping
 * exclude[b,k] (-1 = skip nothing).  Order: logit descending, then id
 * ascending; -0.0 equals +0.0.
 *   draft_logits [B, K+1, V] dtype (device)
 *   exclude      [B, K+1] int32 (device)
 *   fanout       K+1 ints, HOST array, 0 <= F_k <= min(SPV_MAX_FANOUT, V-1)
 *   K+1 <= SPV_MAX_FANOUT_ROWS
 *   V            <= 1,048,576 (else SPV_ERR_UNSUPPORTED: the row merge
 *                holds up to 1,024 per-block candidate lists)
 *   out_ids      [B, sum_k F_k] int32 out (device), k-major then rank
 *   row_status   [B, K+1] int32 out, optional: SPV_ERR_BAD_ROW for NaN rows
 *                (their ids are -1)
 *   workspace    >= spv_fanout_workspace_bytes(B, K, V, max F_k) bytes
 *                (zero-filled once, as for spv_verify_chain).
 */
spv_status spv_fanout_topk(const void *draft_logits, spv_dtype dtype, const int32_t *exclude,
                           const int32_t *fanout, int B, int K, int V,
                           int32_t *out_ids, int32_t *row_status,
                           void *workspace, size_t workspace_bytes, void *stream);

size_t spv_fanout_workspace_bytes(int B, int K, int V, int max_fanout);

/* [SSD] "Core Technical Barrier" (Theorem 12): F_0 * a^(k/(1+r)), unrounded. */
double spv_fanout_size(int F0, double a, double r, int k);

/*
 * spv_fanout_sizes -- the integer fan-out of [SSD] "Core Technical Barrier"
 * (Theorem 12) for positions k = 0..K: F_k = F_0 * a^(k/(1+r)) rounded half
 * away from zero (the page gives the real-valued law; the rounding is this
 * library's reading) and clamped to [0, V-1] (at most V-1 ids remain once
 * the verified token is excluded).  Host function, no CUDA call.
 *   F0 >= 0, a > 0 finite, r > -1 finite, 0 <= K < SPV_MAX_FANOUT_ROWS, V >= 2
 *   out   K+1 int32, HOST array
 * Returns SPV_OK, or SPV_ERR_INVALID_ARG (out untouched).  The result can be
 * passed to spv_fanout_topk when every F_k <= SPV_MAX_FANOUT.
 */
spv_status spv_fanout_sizes(int F0, double a, double r, int K, int V, int32_t *out);

/* Reads the device error word of a workspace (synchronises `stream`):
 * SPV_OK, or SPV_ERR_TIMEOUT if a bounded wait in an earlier call gave up. */
spv_status spv_workspace_status(const void *workspace, void *stream);

/*
 * spv_selftest_timeout -- self-test of the failure path of the bounded waits
 * (no counterpart on the pages).  Every wait of the library's kernels on
 * another CTA's progress gives up after a bounded number of polls, records
 * SPV_ERR_TIMEOUT in the workspace's error word and returns, leaving the
 * CUDA context usable.  This enqueues one small kernel that runs the same
 * bounded wait on header word 1 of `workspace` (cleared first, never set),
 * so it gives up after `polls` polls (each a global load and a short
 * sleep) and records SPV_ERR_TIMEOUT; spv_workspace_status then reports it.
 *   workspace        device memory, 256-byte aligned, >= 256 bytes; its
 *                    header words 0 and 1 are overwritten
 *   polls            1 .. 2^24
 * Returns SPV_OK once enqueued.
 */
spv_status spv_selftest_timeout(void *workspace, size_t workspace_bytes, unsigned polls, void *stream);

/* Human-readable name of a status code (static string). */
const char *spv_status_string(spv_status s);

#ifdef __cplusplus
}
#endif
#endif /* SPV_H */
