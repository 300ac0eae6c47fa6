/*
 * kda.h -- C ABI of the GB300 (sm_103a) gated delta-rule library (libkda.so).
 *
 * The library computes the gated delta rule behind DeltaNet, Gated DeltaNet
 * and Kimi Delta Attention (KDA), one level below the token mixer's
 * projections.  For each (batch, head), with column vectors, a state
 * S in R^{dk x dv} (row i belongs to key channel i) and t = 0 .. T-1:
 *
 *     a_t = exp(-exp(log_alpha_t))            per key channel, per token, or 1
 *     S   = (I - beta_t k_t k_t^T) Diag(a_t) S + beta_t k_t v_t^T
 *     o_t = S^T q_t                           read-out after the write
 *
 * Sources, by page title and section:
 *  - delta rule, read / correct / write, read-out without a normaliser:
 *    "22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 5.2.
 *  - gated form S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T:
 *    "22580: From GPT-2 to Kimi3, Explained" (zharfai.com), "Gated DeltaNet
 *    adds controlled forgetting"; decay applied first for a per-channel a_t.
 *  - per-channel decay alpha = exp(-exp(log_alpha)): "22580: From GPT-2 to
 *    Kimi K3, Explained" (lukebest.github.io), "KDA (per-channel alpha)".
 *  - the chunk-wise parallel form (WY representation, forward substitution on
 *    a C x C unit lower-triangular matrix, W = T K_beta, U = T V_beta, then a
 *    sequential pass over chunks): "22,580: From GPT-2 to Kimi K3"
 *    (yichencityu.github.io), section 6.3.
 *  - the state is the cache handed from call to call ("state in, state out"):
 *    same page, section 5.2, forward(x, cache) -> (o, S).
 *
 * Conventions for every entry point
 *  - All tensors are dense, contiguous, row-major, in DEVICE memory unless
 *    stated; the caller allocates and owns them.  The library allocates no
 *    device memory and keeps no state between calls.
 *  - Every device pointer must be 16-byte aligned; the workspace 256-byte
 *    aligned.  Misaligned pointers return KDA_ERR_INVALID_ARG.
 *  - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *    never synchronise, except kda_chunk_fwd_status.  Arguments are checked
 *    before anything is launched; on an error status nothing was launched.
 *  - Outputs must not overlap inputs, except as stated (h0 == hT; the decode
 *    state is updated in place).
 *  - No C++ exception crosses this interface.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so that including this
 * header needs no CUDA include path. */
struct CUstream_st;
typedef struct CUstream_st *kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative size, bad enum */
  KDA_ERR_UNSUPPORTED = 2, /* valid but outside the supported shapes */
  KDA_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed */
  KDA_ERR_TIMEOUT = 4      /* a bounded on-device wait expired (see kda_chunk_fwd_status) */
} kda_status;

/* Storage type of q, k, v and o.  beta, log_alpha, h0, hT and the decode
 * state are always float32. */
typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Decay mode, i.e. the shape of log_alpha. */
typedef enum {
  KDA_ALPHA_NONE = 0,    /* a = 1 (DeltaNet); log_alpha must be NULL        */
  KDA_ALPHA_SCALAR = 1,  /* one value per token and head (Gated DeltaNet)   */
  KDA_ALPHA_CHANNEL = 2  /* one value per token, head and key channel (KDA) */
} kda_alpha_mode;

/* Implementation choice for kda_chunk_fwd_ex. */
typedef enum {
  KDA_PATH_AUTO = 0,     /* tensor-core path where supported, else CUDA cores */
  KDA_PATH_CUDA_CORE = 1,/* fp32 FFMA chunked kernel (every supported shape)   */
  KDA_PATH_TENSOR = 2,   /* tcgen05 prep + scan (bf16, C = 64, dk = dv in {64,128});
                            KDA_ERR_UNSUPPORTED elsewhere; the scan kernel is
                            chosen as below                                     */
  KDA_PATH_TENSOR_SPLIT_SCAN = 3, /* tensor path, the scan split by value columns
                            (several CTAs per head; the only scan at dk = 64)   */
  KDA_PATH_TENSOR_WIDE_SCAN = 4,  /* tensor path, one scan CTA per (batch, head)
                            holding all value columns (dk = dv = 128 only, else
                            KDA_ERR_UNSUPPORTED).  KDA_PATH_AUTO / _TENSOR use
                            the split scan                                       */
  KDA_PATH_TENSOR_PIPELINED = 5   /* tensor path in up to 16 segments of the
                            sequence (at least 8 chunks each): the prep of
                            segment g + 1 runs beside the one-CTA-per-head scan
                            of segment g, each launch a programmatic dependent
                            of the one before on the caller's stream; the last
                            segment's scan is the split scan.  To the caller's
                            stream the call is ordinary: its first launch waits
                            for earlier work and nothing enqueued after it
                            starts before its last kernel ends.  dk = dv = 128,
                            not the normalised linear-attention rule (else
                            KDA_ERR_UNSUPPORTED); results as the other tensor
                            paths.  Fewer than 16 chunks: one segment         */
} kda_path;

/* ABI version of this header; kda_abi_version() returns the library's. */
#define KDA_ABI_VERSION 1
int kda_abi_version(void);

/* Human-readable name of a status; never NULL; static storage. */
const char *kda_status_string(kda_status s);

/*
 * Bytes of device workspace kda_chunk_fwd needs for this problem (>= 256).
 * Returns 0 if the arguments are invalid or unsupported.  The workspace holds
 * a device error word (first 256 bytes) and, on the tensor-core path, the
 * per-chunk intermediates of the prep kernel (corrected keys and values,
 * decayed queries, the intra-chunk mask and decay factors: 98,816 bytes per
 * (head, chunk) at d = 128, followed at d = 128 by 768 bytes per (head,
 * chunk) that only the normalised linear-attention rule fills, and by one
 * float32 dk x dv state per head that carries the state between the segments
 * of a pipelined call when hT is NULL, and by 256 bytes of work counters that
 * every call resets on its stream).
 */
size_t kda_chunk_fwd_workspace_size(int B, int H, int T, int dk, int dv, int C,
                                    kda_dtype dt, kda_alpha_mode am);
size_t kda_chunk_fwd_workspace_size_ex(int B, int H, int T, int dk, int dv, int C,
                                       kda_dtype dt, kda_alpha_mode am, kda_path path);

/*
 * Chunk-wise parallel prefill of the gated delta rule ("22,580: From GPT-2 to
 * Kimi K3" (yichencityu.github.io), section 6.3, extended with the cumulative
 * per-channel decay).
 *
 *   q, k      [B, H, T, dk]  dtype dt            (device)
 *   v         [B, H, T, dv]  dtype dt            (device)
 *   beta      [B, H, T]      float32             (device)
 *   log_alpha [B, H, T] (SCALAR) or [B, H, T, dk] (CHANNEL) float32, NULL for NONE
 *   h0        [B, H, dk, dv] float32, or NULL for a zero initial state
 *   o         [B, H, T, dv]  dtype dt            (device, written)
 *   hT        [B, H, dk, dv] float32, or NULL    (device, written; may equal h0)
 *   B, H >= 0; T >= 0 (any length: a partial last chunk is handled);
 *   dk, dv in {16, 32, 64, 128}; C in {16, 32, 64} (chunk length);
 *   workspace: >= kda_chunk_fwd_workspace_size(...) bytes of device memory,
 *   256-byte aligned, owned by the caller, not shared with a concurrent call.
 *   Its first 256 bytes are the device error word: they must be zero before
 *   the first call that uses the workspace (cudaMemset them once after
 *   allocating it); the library never clears them itself except through
 *   kda_chunk_fwd_status, which reads and clears them.  A workspace whose
 *   first bytes hold leftover data makes the next kda_chunk_fwd_status
 *   report an error that no call made (and clear it); the rest of the
 *   workspace needs no initialisation.
 *
 * No scaling is applied to q.k (the caller normalises q and k).  o_t includes
 * token t's own write.  Precision: the CUDA-core path computes in float32;
 * the tensor path uses bf16 operands with float32 accumulation and a float32
 * state.  Returns KDA_OK once the work is enqueued.  Device-side failures
 * (a bounded wait that expired) are reported by kda_chunk_fwd_status.
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *beta, const float *log_alpha,
                         const float *h0, void *o, float *hT,
                         int B, int H, int T, int dk, int dv, int C,
                         kda_dtype dt, kda_alpha_mode am,
                         void *workspace, size_t workspace_bytes,
                         kda_stream_t stream);

/*
 * kda_chunk_fwd with an explicit implementation choice and optional launch
 * timing.  `events` (may be NULL when n_events == 0) holds cudaEvent_t
 * handles created by the caller; when n_events >= launches + 1 (launches =
 * kda_chunk_fwd_launches(...)), events[i] is recorded on `stream` just before
 * kernel launch i and events[launches] after the last one, so the caller can
 * time each kernel of the call.  Recording changes no work.  Fewer events
 * than needed: KDA_ERR_INVALID_ARG.
 */
kda_status kda_chunk_fwd_ex(const void *q, const void *k, const void *v,
                            const float *beta, const float *log_alpha,
                            const float *h0, void *o, float *hT,
                            int B, int H, int T, int dk, int dv, int C,
                            kda_dtype dt, kda_alpha_mode am,
                            void *workspace, size_t workspace_bytes,
                            kda_stream_t stream, kda_path path,
                            void *const *events, int n_events);

/* Number of kernel launches one kda_chunk_fwd_ex call makes for this problem
 * (0 for an empty problem), or -1 if the arguments are invalid/unsupported. */
int kda_chunk_fwd_launches(int B, int H, int T, int dk, int dv, int C,
                           kda_dtype dt, kda_alpha_mode am, kda_path path);

/* Name of kernel launch `i` of such a call (static storage), or NULL. */
const char *kda_chunk_fwd_kernel_name(int B, int H, int T, int dk, int dv, int C,
                                      kda_dtype dt, kda_alpha_mode am,
                                      kda_path path, int i);

/*
 * kda_chunk_fwd without a caller-provided workspace, for callers that cannot
 * allocate device memory: code behind a plugin or host interface that is
 * handed only its input and output buffers, or a serving loop that must not
 * call cudaMalloc on its hot path because the call can synchronise the
 * device.  The pages describe no such entry point; it has no counterpart
 * there.
 *
 * Same arguments, meaning and results as kda_chunk_fwd, minus the workspace.
 * The scratch lives in one fixed 64 MiB array inside the library (a
 * file-scope __device__ array that every GPU which loads libkda holds until
 * the process exits).  Problems whose kda_chunk_fwd_workspace_size exceeds
 * 64 MiB (67108864 bytes) are rejected with KDA_ERR_UNSUPPORTED before
 * anything is launched; for the d = 128 tensor path that is about 740
 * (head, 64-token chunk) pairs, e.g. B*H = 8 heads of up to 5,888 tokens.
 * Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * The first call on a device looks up the array's device address on the
 * device that is current at the time (once per device; the device of
 * `stream` must be the current device); make that first call before any
 * stream capture.  Every call clears the array's error word and overwrites
 * the records it uses, but all calls share the one array: calls whose
 * kernels overlap on the GPU (other streams, other host threads) race on it
 * and give undefined results; serialise them.  Device-side wait timeouts are
 * recorded in the shared error word only and are not reported by this call.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *beta, const float *log_alpha,
                                 const float *h0, void *o, float *hT,
                                 int B, int H, int T, int dk, int dv, int C,
                                 kda_dtype dt, kda_alpha_mode am,
                                 kda_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error word of
 * `workspace`.  KDA_OK if every call enqueued with this workspace finished
 * normally; KDA_ERR_TIMEOUT if an on-device wait gave up (the outputs of that
 * call are then undefined); KDA_ERR_CUDA if the synchronisation failed.
 */
kda_status kda_chunk_fwd_status(void *workspace, kda_stream_t stream);

/*
 * kda_chunk_fwd with a choice of update rule and of maps applied to the
 * inputs on the fly (no extra pass over memory).
 *
 * rule:
 *   KDA_RULE_DELTA   the gated delta rule of kda_chunk_fwd.
 *   KDA_RULE_LINEAR  linear attention ("22,580: From GPT-2 to Kimi K3"
 *                    (yichencityu.github.io), section 6.2: the state sums
 *                    k^T v, each query reads the state and its own chunk's
 *                    masked scores), with the same optional decay applied
 *                    first:  S = Diag(a_t) S + k_t v_t^T,  o_t = S^T q_t.
 *                    No normaliser; beta is not read (may be NULL).
 *   KDA_RULE_LINEAR_NORM  the same page's linear attention with its
 *                    normaliser (section 04, "Linear Attention: Bring Back
 *                    the RNN"): a second
 *                    accumulator z = Diag(a_t) z + k_t (the state's column for
 *                    a value of all ones) and o_t = S^T q_t / (q_t . z).  Meant
 *                    with KDA_MAP_QK_ELU1, which keeps q . z positive.  From
 *                    a zero state only: h0 and hT must be NULL
 *                    (KDA_ERR_UNSUPPORTED otherwise); beta is not read.
 * input_maps (bit set), the maps the same page's section 5.2 applies to the
 * projections before the delta rule:
 *   KDA_MAP_QK_SILU_NORM  q, k <- silu(x) / max(||silu(x)||_2, 1e-12) per
 *                         (token, head), silu(x) = x / (1 + exp(-x))
 *   KDA_MAP_BETA_SIGMOID  beta <- 1 / (1 + exp(-beta))   (DELTA only)
 *   KDA_MAP_QK_ELU1       q, k <- elu(x) + 1 = (x > 0 ? x + 1 : exp(x)), the
 *                         feature map of the page's linear attention
 *                         (linear rules only; not with QK_SILU_NORM)
 *
 * Other arguments as kda_chunk_fwd (same workspace size).  rule DELTA with
 * no maps is kda_chunk_fwd (every shape); anything else runs on the tensor
 * path only: bf16, C = 64, dk = dv = 128, else KDA_ERR_UNSUPPORTED.  An
 * unknown rule or map bit, BETA_SIGMOID with a linear rule, QK_ELU1 with the
 * delta rule, or both q, k maps: KDA_ERR_INVALID_ARG.
 */
typedef enum { KDA_RULE_DELTA = 0, KDA_RULE_LINEAR = 1, KDA_RULE_LINEAR_NORM = 2 } kda_rule;
#define KDA_MAP_QK_SILU_NORM 1u
#define KDA_MAP_BETA_SIGMOID 2u
#define KDA_MAP_QK_ELU1 4u
kda_status kda_chunk_fwd_rule(const void *q, const void *k, const void *v,
                              const float *beta, const float *log_alpha,
                              const float *h0, void *o, float *hT,
                              int B, int H, int T, int dk, int dv, int C,
                              kda_dtype dt, kda_alpha_mode am, kda_rule rule,
                              unsigned input_maps, void *workspace, size_t workspace_bytes,
                              kda_stream_t stream);

/*
 * AttnRes depth mixing ("22,580: From GPT-2 to Kimi K3"
 * (yichencityu.github.io), section 12, block_attn_res): for every row r,
 *
 *   K_n = V_n / sqrt(mean_d(V_n^2) + eps)          RMS-normalised keys
 *   a_n = softmax over n of (w . K_n)              over the block axis
 *   h   = sum_n a_n V_n
 *
 *   V   [n_blocks, rows, D]  dtype dt   the stacked block representations
 *   w   [D]                  float32    the learned scoring vector
 *   h   [rows, D]            dtype dt   output
 *
 * The pages' `norm` is read as RMSNorm without a learned scale.  1 <= n_blocks
 * <= 32 and D a multiple of 8 (else KDA_ERR_UNSUPPORTED); eps >= 0; pointers
 * 16-byte aligned.  Arithmetic in float32.  Asynchronous on `stream`.
 */
kda_status kda_attn_res(const void *V, int n_blocks, const float *w, void *h,
                        long long rows, int D, kda_dtype dt, float eps, kda_stream_t stream);

/*
 * kda_chunk_fwd for inputs and outputs in HOST memory, with the transfers
 * overlapped with the prefill.  The pages have no counterpart (they do not
 * discuss where the inputs live); the prefill itself is kda_chunk_fwd.
 *
 *   q, k, v, beta, log_alpha, h0   host, same shapes and types as kda_chunk_fwd
 *   o, hT                          host outputs (hT may be NULL; h0 may be NULL)
 *   group_heads                    0: pipeline steps are segments of the
 *                                  sequence (a chunk-aligned sixteenth of T for
 *                                  every (batch, head) pair; the state is
 *                                  carried from one segment to the next in
 *                                  float32); > 0: steps are groups of that
 *                                  many (batch, head) pairs over all of T
 *   dev_buffer, dev_bytes          device memory, 256-byte aligned, at least
 *                                  kda_chunk_fwd_host_buffer_size(...) bytes,
 *                                  owned by the caller; it holds the shared
 *                                  workspace (its start: read device errors
 *                                  with kda_chunk_fwd_status(dev_buffer, ...);
 *                                  its first 256 bytes must be zero before
 *                                  the first call, as for kda_chunk_fwd)
 *                                  (segments: also the carried state) and two
 *                                  staging slots of one pipeline step
 *
 * While step s runs on `stream`, step s + 1 is copied in and step s - 1
 * copied out on two streams that the call creates and releases (nothing is
 * kept between calls).  Segments leave less work after the last copy-in (one
 * segment's prefill and copy-out instead of one group's whole-sequence scan).
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister): from
 * pageable memory the copies are correct but do not overlap.  The call returns once
 * everything is enqueued; all of it, copies included, completes on `stream`
 * (synchronise `stream` before reading o or hT).  Results equal those of
 * kda_chunk_fwd on device copies of the inputs, bit for bit.  Errors: as
 * kda_chunk_fwd, plus KDA_ERR_INVALID_ARG for a null or misaligned dev_buffer
 * or dev_bytes below the required size; checked before anything is enqueued.
 */
size_t kda_chunk_fwd_host_buffer_size(int B, int H, int T, int dk, int dv, int C,
                                      kda_dtype dt, kda_alpha_mode am, int group_heads);
kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                              const float *beta, const float *log_alpha,
                              const float *h0, void *o, float *hT,
                              int B, int H, int T, int dk, int dv, int C,
                              kda_dtype dt, kda_alpha_mode am, int group_heads,
                              void *dev_buffer, size_t dev_bytes, kda_stream_t stream);

/*
 * One recurrent decode step for N x H independent states, in place
 * ("22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 5.2, with
 * t = 1 and the cached state; decay as in kda_chunk_fwd):
 *
 *   S = Diag(a) S;  u = beta (v - S^T k);  S = S + k u^T;  o = S^T q
 *
 *   q, k      [N, H, dk]  dtype dt
 *   v         [N, H, dv]  dtype dt
 *   beta      [N, H]      float32
 *   log_alpha [N, H] (SCALAR) or [N, H, dk] (CHANNEL) float32, NULL for NONE
 *   S_inout   [N, H, dk, dv] float32, read and overwritten in place
 *   o         [N, H, dv]  dtype dt (written)
 *   N, H >= 0; dk, dv in {16, 32, 64, 128}.
 * The state is read once and written once (float32 arithmetic throughout).
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *beta, const float *log_alpha,
                           float *S_inout, void *o,
                           int N, int H, int dk, int dv,
                           kda_dtype dt, kda_alpha_mode am, kda_stream_t stream);

/*
 * Device self-test of the bounded-wait mechanism: launches one block that
 * waits on an mbarrier nothing will ever complete, with a wait limit of
 * `spin_limit` polls.  The wait gives up, the kernel records
 * KDA_ERR_TIMEOUT in the workspace's error word and returns normally, so the
 * CUDA context stays usable.  Read the result with kda_chunk_fwd_status.
 * spin_limit must be in [1, 1<<20].
 */
kda_status kda_selftest_wait_timeout(void *workspace, size_t workspace_bytes,
                                     unsigned spin_limit, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
