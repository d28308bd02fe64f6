/*
 * spec_verify: batched speculative-decoding verification by rejection
 * sampling, for one NVIDIA GB300 (sm_103a).
 *
 * What is computed (per chain b of k drafted tokens x_1..x_k):
 *   p_i = softmax(target_logits[b, i-1, :] / T_b)   i = 1..k+1   (target rows)
 *   q_i = softmax(draft_logits[b, i-1, :] / T_b)    i = 1..k     (draft rows)
 *   Drafts are accepted or rejected against the target distribution, which
 *   preserves it ("Optimizing speculative decoding", section "Rejection
 *   sampling and a loss that optimizes acceptance directly", first bullet):
 *   x_i is accepted while u_i < min(1, p_i(x_i) / q_i(x_i)).  At the first
 *   rejection (position tau+1) one token is drawn from the normalised residual
 *   max(0, p - q); if all k are accepted, a bonus token is drawn from p_{k+1}
 *   (the k+1-th target row that the single verification pass provides:
 *   "Optimizing speculative decoding", section "The draft model moved
 *   inside").  The final draw uses its own uniform u_{k+1} and the inverse
 *   CDF y = min{ j : u * S < C_j }.  tau is the accepted length (page
 *   "DSpark for GLM-5.2", introduction).  The per-position total-variation
 *   distance 0.5 * sum_j |p_i(j) - q_i(j)| ("Optimizing speculative
 *   decoding", the section above, second bullet) is reported for every
 *   position; 1 - TV is the per-position acceptance probability
 *   sum_j min(p, q) ("Optimizing speculative decoding", section "Kimi K3").
 *   T_b == 0 means greedy: p and q are one-hot on the lowest-index maximum,
 *   so a draft is accepted iff it equals the target argmax.
 *
 * Conventions shared by every entry point:
 *   - Logit tensors are dense, row-major, C-contiguous, in device memory,
 *     element type fp32 (SV_FP32) or bf16 (SV_BF16).  A logit row must
 *     contain no NaN and no +inf; -inf marks a masked token; at least one
 *     entry must be finite; for T > 0, |max logit| / T must stay below
 *     2^22 / log2(e).  A chain that breaks any of these, has a temperature
 *     that is negative, NaN or infinite, or a draft token outside [0, V), is
 *     an invalid chain: its tau is -1 and its tokens are -1 (no fault).
 *   - All pointers are device pointers unless the name says host; the caller
 *     owns every buffer; the library only reads inputs and writes outputs.
 *   - Calls are asynchronous and ordered on the caller's CUDA stream
 *     (`cuda_stream` is a cudaStream_t; NULL = the legacy default stream).
 *     Nothing is returned to the host until the caller synchronises, except
 *     by spec_verify_get_error, which synchronises.
 *   - Argument errors are detected on the host before any launch and
 *     returned as a status; no exception crosses the interface.
 *   - A handle is not thread-safe; use one handle per stream.  Different
 *     handles may run at the same time on different streams: their kernels
 *     can share SMs, and the tensor memory they allocate per CTA (256 or 512
 *     columns, in the larger instances) never exceeds an SM's 512 columns
 *     whatever the mix, so no launch waits on another.
 *   - Uniforms are in [0, 1); the seeded generator used by this project
 *     produces them on the 2^-24 lattice.
 *   - Limits: 1 <= k <= 31; V <= 327680 (bf16) or 163840 (fp32).  Above
 *     163840 (bf16) or 81920 (fp32) the kernels hold twice the registers per
 *     thread and run one CTA per SM instead of two.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spec_verify_ctx* spec_verify_t;

/* Status codes returned by every call. */
enum {
  SV_OK = 0,
  SV_ERR_ARG = 1,     /* null handle/pointer, bad batch size, misaligned array */
  SV_ERR_DTYPE = 2,   /* unknown logit dtype */
  SV_ERR_SIZE = 3,    /* k or V outside the supported range */
  SV_ERR_CUDA = 4,    /* a CUDA runtime call or launch failed */
  SV_ERR_ALLOC = 5,   /* device or host allocation failed in init */
  SV_ERR_DATA = 6,    /* (get_error) some chains were invalid since the last check */
  SV_ERR_TIMEOUT = 7  /* (get_error) a bounded device wait expired: from then until get_error clears
                         the flag, every call reports every chain invalid (tau = -1, TV NaN) */
};

/* Logit element types. */
enum { SV_FP32 = 0, SV_BF16 = 1 };

/* Flags for spec_verify_init. */
enum {
  SV_FLAG_HOST_STAGING = 1u,  /* also allocate device staging for spec_verify_host: max_batch
                                 chains of logits (used only for pageable host logits) and the
                                 small inputs and outputs */
  SV_FLAG_NO_TMA = 2u,        /* load logits with plain loads instead of bulk copies (testing) */
  SV_FLAG_KERNEL_TIMING = 4u  /* record a CUDA event pair around the verification kernel of each call */
};

/* Create a handle for chains of k drafts over a vocabulary of `vocab`
 * tokens with logits of type `logit_dtype`, for batches of up to
 * `max_batch` chains.  Allocates the device workspace (per-position accept
 * decisions, greedy tokens, row statistics and per-range masses: about
 * 552*(k+1) bytes per chain) and, with SV_FLAG_HOST_STAGING, device copies of
 * every input and output for max_batch chains.  Uses the current CUDA device; the handle
 * must be used on that device.  SV_ERR_SIZE also when max_batch*(k+1) reaches
 * 2^31.  Writes NULL to *h on failure. */
int spec_verify_init(spec_verify_t* h, int max_batch, int k, int vocab, int logit_dtype, unsigned flags);

/* Verify `batch` chains (0 <= batch <= max_batch).
 *   target_logits  [batch, k+1, V]  row i is the target distribution after x_1..x_i
 *   draft_logits   [batch, k,   V]  row i is the distribution x_{i+1} was drawn from
 *   draft_tokens   [batch, k]   int32
 *   temperature    [batch]      fp32, one per chain, 0 = greedy
 *   uniforms       [batch, k+1] fp32 in [0,1): u[:, 0..k-1] accept tests,
 *                               u[:, k] the final (residual or bonus) draw
 *   out_tokens     [batch, k+1] int32: x_1..x_tau, then the residual or bonus
 *                               token, then -1 padding
 *   out_tau        [batch]      int32: accepted drafts 0..k (-1: invalid chain)
 *   out_p_draft    [batch, k]   fp32 or NULL: p_i(x_i) for every position
 *                               (NaN where the position's rows, temperature
 *                               or token are invalid)
 *   out_q_draft    [batch, k]   fp32 or NULL: q_i(x_i) for every position (same)
 *   out_tv         [batch, k]   fp32 or NULL: TV distance of every position
 * Integer and fp32 arrays must be 4-byte aligned; logits whose base is
 * 16-byte aligned and whose row size V*sizeof(elem) is a multiple of 16 use
 * bulk (TMA) copies, anything else plain loads.  Two kernel launches. */
int spec_verify(spec_verify_t h, int batch,
                const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                int32_t* out_tokens, int32_t* out_tau,
                float* out_p_draft, float* out_q_draft, float* out_tv,
                void* cuda_stream);

/* Lazy verification: the same protocol, verifying positions in order and
 * reading no logit row past a chain's first rejection (the protocol stops
 * there: "Optimizing speculative decoding", section "The draft model moved
 * inside", and "DSpark for GLM-5.2", introduction).  out_tokens and out_tau
 * are bit-identical to spec_verify's for every chain whose rows up to its
 * stop are valid; a chain is invalid (tau = -1) only if a row it reads is
 * (rows after the stop are never read, so their contents do not matter).
 * There is no p, q or TV output (positions after the stop are not
 * evaluated), and accepted positions skip the residual pass.  Two kernel
 * launches: one walks every chain position by position up to its stop
 * (each cluster of CTAs works on two chains at a time and takes the next
 * chain from a shared counter when one stops), then the finalize kernel
 * draws the final tokens. */
int spec_verify_lazy(spec_verify_t h, int batch,
                     const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                     int32_t* out_tokens, int32_t* out_tau, void* cuda_stream);

/* Training-side losses on the draft-target overlap, and their gradient with
 * respect to the draft logits (the target is frozen).  For position i of a
 * chain (target row i, draft row i, the chain's T > 0):
 *   alpha_i = sum_x min(p_i(x), q_i(x)) = 1 - TV_i, the probability that the
 *   protocol accepts the drafted token ("Optimizing speculative decoding",
 *   section "Kimi K3");
 *   SV_LOSS_TV:      l_i = TV_i = 1 - alpha_i (section "Rejection sampling
 *                    and a loss that optimizes acceptance directly");
 *   SV_LOSS_OVERLAP: l_i = -ln alpha_i (section "Kimi K3").
 * The loss is L = sum_i w_i l_i and the gradient
 *   dL/d draft_i[m] = w_i dl/dalpha (q_i(m)/T) ([q_i(m) < p_i(m)] - beta_i),
 *   beta_i = sum_{x: q_i(x) < p_i(x)} q_i(x),
 * with the strict side taken at p == q (a subgradient).
 *   weights     [batch, k] fp32 or NULL (all 1)
 *   out_loss    [batch, k] fp32 or NULL: l_i (NaN for an invalid position)
 *   grad_draft  [batch, k, V] in the logit dtype (bf16 rounded to nearest
 *               even): every entry written, 0 for an invalid position
 * A position is invalid when T is not > 0 and finite or a row has no finite
 * maximum.  One kernel launch. */
enum { SV_LOSS_TV = 0, SV_LOSS_OVERLAP = 1 };
int spec_verify_loss_grad(spec_verify_t h, int batch,
                          const void* target_logits, const void* draft_logits, const float* temperature,
                          int loss_kind, const float* weights, float* out_loss, void* grad_draft,
                          void* cuda_stream);

/* spec_verify, and also the entropy of every logit row's distribution, in
 * the same pass over the logits.  The pages tie the fall of acceptance to
 * fluctuations in the entropy of the model's output, i.e. in how widely its
 * probability mass is spread ("Optimizing speculative decoding" and "GLM-5.2: Tuning
 * MTP speculative decoding to the limit", section "Rejection sampling and a
 * loss that optimizes acceptance directly"); the statistic here is the
 * Shannon entropy, in nats, of p = softmax(z / T), the distribution the
 * verifier itself uses:
 *   out_entropy_target [batch, k+1] fp32: H of target row i
 *   out_entropy_draft  [batch, k]   fp32: H of draft row i
 * Both NULL (then this is spec_verify) or both non-NULL and 4-byte aligned,
 * else SV_ERR_ARG.  H = 0 for greedy chains (T == 0).  H = NaN for a chain
 * with an invalid temperature, and for a row without a finite maximum.
 * Masked logits (-inf) add nothing.  The other outputs are bit-identical to
 * spec_verify's.  Two kernel launches. */
int spec_verify_ex(spec_verify_t h, int batch,
                   const void* target_logits, const void* draft_logits,
                   const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                   int32_t* out_tokens, int32_t* out_tau,
                   float* out_p_draft, float* out_q_draft, float* out_tv,
                   float* out_entropy_target, float* out_entropy_draft,
                   void* cuda_stream);

/* Allocation-free spec_verify.  The pages have no counterpart of this call;
 * it exists for callers that cannot allocate device memory.  cudaMalloc may
 * synchronise the whole device, and a serving engine that has reserved its
 * memory for the KV cache at start-up may refuse any further allocation, so
 * such callers cannot use spec_verify_init.  This call takes no handle and
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine):
 * its workspace is a file-scope device array of SV_NOALLOC_SCRATCH_BYTES
 * that every GPU loading the library holds until the process exits.
 * Arguments, layouts, outputs and invalid-chain reporting (tau = -1) are
 * those of spec_verify, plus k, vocab and logit_dtype in place of a handle.
 * Limit: the workspace needs about 4*k + 548*(k+1) bytes per chain (4,412 at
 * k = 7), so batch may be up to about 1,900 chains at k = 7 and 950 at
 * k = 15; larger batches return SV_ERR_SIZE before any launch.
 * Notes: the first call on each device does a one-time set-up (looks up the
 * array's device address with cudaGetSymbolAddress, sets kernel attributes,
 * queries occupancy) and should be made before any stream capture.  All
 * calls share the one array and its contents persist between calls (the
 * counters that must start at zero are cleared on the stream at each call),
 * so calls that overlap on the GPU, on different streams, race with each
 * other: order them on one stream.  Counters are not reported: invalid
 * chains show up as tau = -1, and a bounded device wait that gives up during
 * a call makes that call report every chain invalid (tau = -1, TV NaN). */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
int spec_verify_noalloc(int batch, int k, int vocab, int logit_dtype,
                        const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                        int32_t* out_tokens, int32_t* out_tau,
                        float* out_p_draft, float* out_q_draft, float* out_tv,
                        void* cuda_stream);

/* Per-position TV distance only: out_tv[b, i] = 0.5 * sum_j |p_{i+1}(j) - q_{i+1}(j)|
 * for the k target/draft row pairs of each chain (the target's bonus row is
 * not read).  A position whose rows or temperature are invalid gets NaN.
 * Two kernel launches. */
int spec_verify_tv(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                   const float* temperature, float* out_tv, void* cuda_stream);

/* spec_verify for callers whose inputs and outputs live in host memory.
 * Same arguments and layouts as spec_verify, but every pointer is a host
 * pointer; the handle must have been created with SV_FLAG_HOST_STAGING.
 * Logits in page-locked memory that the device can address (pinned memory on
 * a system with unified addressing) are read in place by the kernels over the
 * host link; other logits are first copied into the handle's device staging.
 * The small inputs go through the staging, and the outputs are copied back,
 * all on `cuda_stream`.  The call returns after enqueueing (synchronise the
 * stream before reading outputs); the host buffers must stay valid until then. */
int spec_verify_host(spec_verify_t h, int batch,
                     const void* host_target_logits, const void* host_draft_logits,
                     const int32_t* host_draft_tokens, const float* host_temperature,
                     const float* host_uniforms,
                     int32_t* host_out_tokens, int32_t* host_out_tau,
                     float* host_out_p_draft, float* host_out_q_draft, float* host_out_tv,
                     void* cuda_stream);

/* Synchronise the device and report what the kernels flagged since the last
 * call: SV_OK, SV_ERR_DATA (with the number of invalid chains in
 * *invalid_count if non-NULL), SV_ERR_TIMEOUT, or SV_ERR_CUDA.  Clears the
 * flags. */
int spec_verify_get_error(spec_verify_t h, int* invalid_count);

/* Self-test of the bounded device waits (for tests).  One thread waits on a
 * shared-memory barrier that nothing completes, first with the kernels' stage
 * wait and then with their cluster-scope wait, each limited to `polls` polls
 * (the kernels use 2^18, about one second).  The first wait must give up and set the handle's
 * timeout flag; the second must then see the flag and return early.  Nothing
 * is left in flight, so the context stays usable.  Synchronises, stores the
 * SM clock cycles each wait took in elapsed_cycles[0..1] (nullable), and
 * returns the handle's status without clearing it: SV_ERR_TIMEOUT when the
 * waits expired as they should.  The flag then stays set, as after a real
 * timeout, so calls on the handle report every chain invalid until
 * spec_verify_get_error clears it.  SV_ERR_ARG for polls < 1. */
int spec_verify_selftest_wait(spec_verify_t h, int polls, long long* elapsed_cycles);

/* Launch geometry chosen at init: vocabulary slices per row (thread-block
 * cluster size), persistent clusters, register rounds per thread, whether
 * bulk copies are enabled, and kernel launches per spec_verify call.
 * Any pointer may be NULL. */
int spec_verify_info(spec_verify_t h, int* cluster_size, int* n_clusters, int* rounds, int* tma,
                     int* launches_per_call);

/* With SV_FLAG_KERNEL_TIMING: wait for the recorded events and write the
 * duration in milliseconds of the verification kernel (the first of the
 * two launches of spec_verify, or the only launch of spec_verify_tv) of up
 * to max_n calls made since the previous read into out_ms, oldest first;
 * *n_out receives the count.  At most 4096 calls are recorded between reads.
 * Returns SV_ERR_ARG if the handle was created without the flag. */
int spec_verify_kernel_times(spec_verify_t h, float* out_ms, int max_n, int* n_out);

/* Free the handle and its device memory (NULL is a no-op). */
void spec_verify_destroy(spec_verify_t h);

/* Static description of a status code. */
const char* spec_verify_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
