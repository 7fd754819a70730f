/*
 * lce.h -- C ABI of the fused linear cross-entropy library (liblce.so) for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation is the loss at the end of a language model, as defined in
 * "Training Beyond 1M Tokens" (TRL guide), section "The loss is the first
 * thing to break": the last hidden states h (L x H) are multiplied by the
 * LM-head weights W (V x H, nn.Linear layout) into logits z = h W^T (L x V),
 * and the loss is the cross entropy of those logits against the integer
 * labels. Section "The massive logits matrix: chunk it" of the same guide
 * gives the reason the logits are never materialised: the loss is a sum over
 * rows and each softmax runs along one row's vocabulary, so rows can be
 * processed piecewise. This library goes further than row pieces: the
 * forward keeps only running per-row (max, sum of exp) statistics in the
 * tensor-core epilogue; the backward recomputes the logits one bounded row
 * chunk at a time. Extra device memory is O(chunk_rows * V), never O(L * V).
 *
 * Definition (the reduction is this library's reading; the pages only say
 * the per-row pieces are summed):
 *   valid(i)  = labels[i] != ignore_index and 0 <= labels[i] < V
 *   N         = #{i : valid(i)}
 *   lse[i]    = log sum_j exp(z[i][j])                     (every row)
 *   loss      = (1/N) sum_{valid i} (lse[i] - z[i][labels[i]]),  0 if N = 0
 *   G[i][j]   = dloss/N (exp(z[i][j] - lse[i]) - [j == labels[i]]), valid i
 *             = 0                                               otherwise
 *   dH        = G W,   dW = G^T h
 *
 * Conventions shared by every call below:
 *   - All pointers named "device" are CUDA device pointers owned by the
 *     caller; the library allocates nothing and keeps no pointer after the
 *     call returns (work is queued on `stream`).
 *   - Matrices are row-major and contiguous. h, W, dH and the workspace must
 *     be 16-byte aligned, and H must be a multiple of 8 (the TMA copy
 *     engine needs 16-byte row strides).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Calls are asynchronous on that stream; none synchronises the host,
 *     except lce_get_error.
 *   - Argument errors are returned synchronously, before anything is
 *     queued. Errors found on the device (a label out of range, a bounded
 *     wait that expired) set the library's device error word, read by
 *     lce_get_error; the kernels never trap.
 *   - Inputs of dtype LCE_F32 are rounded to bf16 on the device (into the
 *     workspace) before the tensor-core contractions; accumulation is fp32.
 *   - Results are deterministic: no floating-point atomics; fixed reduction
 *     orders for a fixed shape, dtype and chunk_rows.
 *   - The functions are thread-safe for distinct workspaces; calls that
 *     share a workspace must be ordered on one stream. The device is the
 *     calling thread's current one; a thread with no CUDA context current
 *     yet gets its current device's primary context made current by the
 *     first call (a context the caller made current is kept).
 */
#ifndef LCE_H_
#define LCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LCE_OK = 0,
  LCE_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment */
  LCE_ERR_UNSUPPORTED = 2, /* device is not sm_103, or unknown dtype */
  LCE_ERR_WORKSPACE = 3,   /* ws_bytes below lce_workspace_size() */
  LCE_ERR_LABEL_RANGE = 4, /* a label outside [0, V) that is not ignore_index
                              (that row was treated as ignored) */
  LCE_ERR_TIMEOUT = 5,     /* a bounded wait inside a kernel expired */
  LCE_ERR_CUDA = 6         /* a CUDA runtime call failed */
} lce_status;

typedef enum {
  LCE_BF16 = 0, /* h, W (and dH) are bfloat16 */
  LCE_F32 = 1   /* h, W (and dH) are float32; computed from bf16 roundings */
} lce_dtype;

/*
 * Bytes of device workspace that lce_forward and lce_backward need for this
 * shape (the same buffer serves both). chunk_rows is the backward's row
 * chunk (0 = the library's default). Returns 0 for invalid sizes.
 * The dominant term is chunk_rows * round_up(V, 8) * 2 bytes (the bf16
 * gradient-logit chunk); with LCE_F32 add bf16 copies of h and W.
 * lce_forward and lce_forward_slice use only the regions before the
 * gradient-logit chunk, so any chunk_rows gives them enough.
 */
size_t lce_workspace_size(int64_t L, int64_t H, int64_t V, lce_dtype dt,
                          int64_t chunk_rows);

/* The row chunk the backward uses when chunk_rows = 0. */
int64_t lce_default_chunk_rows(int64_t L, int64_t H, int64_t V);

/*
 * Forward. Source: "Training Beyond 1M Tokens", sections "The loss is the
 * first thing to break" and "The massive logits matrix: chunk it".
 *   h       device, [L][H] of dt
 *   W       device, [V][H] of dt
 *   labels  device, [L] int64
 *   loss    device, [1] float32 out: mean loss over valid rows (0 if none)
 *   lse     device, [L] float32 out: per-row log-sum-exp (every row); keep
 *           it for lce_backward
 *   ws      device workspace of ws_bytes >= lce_workspace_size(...)
 * Queues: label count, one persistent tensor-core kernel over all logit
 * tiles (online log-sum-exp + label-logit gather in its epilogue), a
 * per-row combine, a one-block loss reduction.
 */
lce_status lce_forward(const void* h, const void* W, lce_dtype dt,
                       const int64_t* labels, int64_t L, int64_t H, int64_t V,
                       int64_t ignore_index, float* loss, float* lse, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * Backward. The pages do not describe it; it is the gradient of the forward
 * above: G = dloss/N (softmax - onehot) on valid rows.
 *   lse        device, [L] float32 from lce_forward on the same inputs
 *   dloss      device, [1] float32: gradient of the scalar loss
 *   chunk_rows rows per chunk (multiple of 128, or 0 for the default)
 *   dH         device, [L][H] of dt, overwritten
 *   dW         device, [V][H] float32, overwritten
 *   Either of dH, dW may be NULL (not both): that gradient is not computed
 *   and its contraction is skipped (a frozen head: dW NULL, about a third
 *   of the backward's flops saved); the other is the same, bit for bit.
 * For each chunk of rows: one tensor-core kernel recomputes the chunk's
 * logits and writes bf16 (softmax - onehot) into the workspace, one computes
 * the chunk's dH rows, one adds the chunk's contribution into dW (fp32
 * read-add-write, chunks in order, no atomics).
 */
lce_status lce_backward(const void* h, const void* W, lce_dtype dt,
                        const int64_t* labels, const float* lse, int64_t L,
                        int64_t H, int64_t V, int64_t ignore_index,
                        const float* dloss, int64_t chunk_rows, void* dH,
                        float* dW, void* ws, size_t ws_bytes, void* stream);

/*
 * Forward and backward in one call, without recomputing the logits: for
 * each row chunk, one tensor-core kernel computes the chunk's logits once
 * and writes, besides the forward's per-row statistics, each 256-column
 * tile's row maximum and the bf16 exponentials relative to it into the
 * workspace; once the chunk's lse is known, a memory-bound pass turns them
 * in place into softmax - onehot, which feeds the same dH and dW
 * contractions as lce_backward. Executes 6 L H V flops instead of the
 * 8 L H V of lce_forward + lce_backward, for about 6 bytes of extra HBM
 * traffic per logit. Not on the pages, which describe only the forward's
 * chunking ("Training Beyond 1M Tokens", section "The massive logits
 * matrix: chunk it").
 *   Arguments as lce_forward and lce_backward; loss, lse, dH and dW are all
 *   outputs, the gradients being those of the loss itself (dloss = 1).
 *   Scale them afterwards with lce_scale_gradients for another dloss.
 *   dH and dW may each be NULL: that gradient's contraction is skipped
 *   (both NULL: only the forward's outputs, from the fused logits pass).
 * The softmax is rounded to bf16 as exp(z - tile max) before being
 * rescaled, so G differs from lce_backward's by bf16 rounding only.
 */
lce_status lce_forward_backward(const void* h, const void* W, lce_dtype dt,
                                const int64_t* labels, int64_t L, int64_t H,
                                int64_t V, int64_t ignore_index,
                                int64_t chunk_rows, float* loss, float* lse,
                                void* dH, float* dW, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * dH *= dloss[0] and dW *= dloss[0] in place (dH of dtype dt, [L][H]; dW
 * fp32 [V][H]; dloss a device float; either gradient may be NULL and is
 * then left out). Nothing is done when dloss[0] is exactly 1. For gradients from lce_forward_backward under another upstream
 * gradient; bf16 dH is rounded again after the multiply.
 */
lce_status lce_scale_gradients(void* dH, lce_dtype dt, int64_t L, int64_t H,
                               float* dW, int64_t V, const float* dloss,
                               void* stream);

/*
 * Loss variants: label smoothing and z-loss. No counterpart on the pages,
 * which define only the plain cross entropy ("Training Beyond 1M Tokens",
 * section "The loss is the first thing to break"); both are common
 * companions of it in language-model training. For every row that takes
 * part, with q_j = (1 - label_smoothing) [j == y_i] + label_smoothing / V:
 *   loss_i = sum_j q_j (lse_i - z_ij) + z_loss * lse_i^2
 *          = lse_i - (1 - eps) z_{i,y_i} - (eps / V) sum_j z_ij
 *            + z_loss * lse_i^2                     (eps = label_smoothing)
 *   loss   = (1/N) sum_{valid i} loss_i               (0 if N = 0)
 *   G_ij   = dloss/N ((1 + 2 z_loss lse_i) softmax_ij - q_j)
 * Ignored rows add nothing, as in the plain loss. Fields:
 *   label_smoothing  in [0, 1]; 0 = the one-hot target
 *   z_loss           >= 0, with 2 * z_loss finite in float; 0 = no z-loss
 * Other values return LCE_ERR_INVALID_ARG before anything is queued.
 * A NULL pointer or {0, 0} is the plain loss, computed with exactly the
 * arithmetic of the calls without options (the same bits). Label smoothing
 * makes the forward keep, per row and column split, the sum of the logits
 * as well (a workspace region that lce_workspace_size always counts).
 */
typedef struct {
  float label_smoothing;
  float z_loss;
} lce_loss_opts;

/* lce_forward, lce_backward and lce_forward_backward with a loss variant
 * (opts may be NULL); every other argument as in the call without _ex.
 * lce_backward_ex must be given the opts of the lce_forward_ex whose lse it
 * uses (lse itself does not depend on them). */
lce_status lce_forward_ex(const void* h, const void* W, lce_dtype dt,
                          const int64_t* labels, int64_t L, int64_t H,
                          int64_t V, int64_t ignore_index,
                          const lce_loss_opts* opts, float* loss, float* lse,
                          void* ws, size_t ws_bytes, void* stream);
lce_status lce_backward_ex(const void* h, const void* W, lce_dtype dt,
                           const int64_t* labels, const float* lse, int64_t L,
                           int64_t H, int64_t V, int64_t ignore_index,
                           const lce_loss_opts* opts, const float* dloss,
                           int64_t chunk_rows, void* dH, float* dW, void* ws,
                           size_t ws_bytes, void* stream);
lce_status lce_forward_backward_ex(const void* h, const void* W, lce_dtype dt,
                                   const int64_t* labels, int64_t L, int64_t H,
                                   int64_t V, int64_t ignore_index,
                                   const lce_loss_opts* opts,
                                   int64_t chunk_rows, float* loss, float* lse,
                                   void* dH, float* dW, void* ws,
                                   size_t ws_bytes, void* stream);

/*
 * Vocabulary-parallel form (several processes each hold a slice of the
 * head's rows, W[v0 .. v0 + Vs) of a vocabulary of V_total, and all of h).
 * "Training Beyond 1M Tokens", section "The massive logits matrix: chunk
 * it", explains that rows split cleanly because the softmax runs along one
 * row's vocabulary; splitting the vocabulary instead needs, per row, each
 * slice's maximum logit m and sum of exp(z - m), merged exactly as
 * lse = M + ln sum_r s_r exp(m_r - M), M = max_r m_r. Three calls:
 *
 * lce_forward_slice: one slice's statistics.
 *   h        device [L][H] of dt (every row)
 *   W        device [Vs][H] of dt: rows v0 .. v0 + Vs - 1 of the head
 *   labels   device [L] int64, ids of the whole vocabulary
 *   v0, Vs, V_total   0 <= v0, v0 + Vs <= V_total
 *   m, s     device [L] float32 out: max_j z_ij and sum_j exp(z_ij - m_i)
 *            over the slice's columns j
 *   zy       device [L] float32 out: z_{i, y_i} where y_i lies in the slice
 *            and takes part, else 0 (so the slices' values sum to it)
 *   ws       workspace of lce_workspace_size(L, H, Vs, dt, chunk_rows)
 * Labels outside [0, V_total) that are not ignore_index raise
 * LCE_ERR_LABEL_RANGE (the row is ignored everywhere).
 */
lce_status lce_forward_slice(const void* h, const void* W, lce_dtype dt,
                             const int64_t* labels, int64_t L, int64_t H,
                             int64_t Vs, int64_t v0, int64_t V_total,
                             int64_t ignore_index, float* m, float* s,
                             float* zy, void* ws, size_t ws_bytes,
                             void* stream);

/*
 * lce_combine_slices: the P slices' statistics, gathered by the caller into
 * m, s, zy (device [P][L] float32 each, slice r at offset r * L, any slice
 * order as long as every process uses the same), merged per row in slice
 * order into lse (device [L] float32 out) and the mean loss over valid rows
 * (device [1] float32 out, 0 if none). ws: device, 16-byte aligned, at least
 * lce_combine_workspace_size(L) bytes (any slice call's workspace is
 * larger). Every process that runs it on the same gathered input gets the
 * same bits.
 */
size_t lce_combine_workspace_size(int64_t L);
lce_status lce_combine_slices(const float* m, const float* s, const float* zy,
                              int64_t P, const int64_t* labels, int64_t L,
                              int64_t V_total, int64_t ignore_index,
                              float* loss, float* lse, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * lce_backward_slice: one slice's share of the backward, given the merged
 * lse: G_s = dloss/N (exp(z - lse) - [j == y]) over the slice's columns
 * (N counted over the whole vocabulary's valid labels), recomputing the
 * logits chunk by chunk as lce_backward does.
 *   dH_part  device [L][H] float32 out: G_s W_s; the sum over the slices is
 *            dH (the caller's all-reduce)
 *   dW       device [Vs][H] float32 out: this slice's rows of dW
 *   either of dH_part, dW may be NULL (not both), as in lce_backward
 *   other arguments as lce_forward_slice and lce_backward
 */
lce_status lce_backward_slice(const void* h, const void* W, lce_dtype dt,
                              const int64_t* labels, const float* lse,
                              int64_t L, int64_t H, int64_t Vs, int64_t v0,
                              int64_t V_total, int64_t ignore_index,
                              const float* dloss, int64_t chunk_rows,
                              float* dH_part, float* dW, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * The same vocabulary slice without recomputing its logits in the backward
 * (the recompute-free form of lce_forward_backward, split at the exchange):
 * lce_forward_slice_exp returns what lce_forward_slice returns and also
 * keeps, in ws, each row's bf16 exponentials relative to each 256-column
 * tile's maximum and those maxima; after the caller has merged the slices'
 * statistics into lse (lce_combine_slices), lce_backward_slice_exp turns
 * them in place into G_s = dloss/N (softmax - onehot) and computes dH_part
 * (fp32 [L][H], summed over the slices by the caller) and the slice's dW
 * (fp32 [Vs][H], written, not accumulated). Executes 6 L H Vs flops per
 * slice instead of the 8 L H Vs of lce_forward_slice + lce_backward_slice,
 * for L x round_up(Vs, 8) x 2 bytes of workspace (5 GB for L = 131072 rows
 * and a 151936 / 8 slice).
 *   ws  lce_slice_exp_workspace_size(L, H, Vs, dt) bytes, the same buffer
 *       for both calls and untouched in between; other arguments as
 *       lce_forward_slice and lce_backward_slice (dH_part or dW may be
 *       NULL, not both).
 */
size_t lce_slice_exp_workspace_size(int64_t L, int64_t H, int64_t Vs,
                                    lce_dtype dt);
lce_status lce_forward_slice_exp(const void* h, const void* W, lce_dtype dt,
                                 const int64_t* labels, int64_t L, int64_t H,
                                 int64_t Vs, int64_t v0, int64_t V_total,
                                 int64_t ignore_index, float* m, float* s,
                                 float* zy, void* ws, size_t ws_bytes,
                                 void* stream);
lce_status lce_backward_slice_exp(const void* h, const void* W, lce_dtype dt,
                                  const int64_t* labels, const float* lse,
                                  int64_t L, int64_t H, int64_t Vs, int64_t v0,
                                  int64_t V_total, int64_t ignore_index,
                                  const float* dloss, float* dH_part,
                                  float* dW, void* ws, size_t ws_bytes,
                                  void* stream);

/*
 * The vocabulary-parallel calls with a loss variant (lce_loss_opts; NULL or
 * {0, 0} is the plain loss, with the same bits as the calls without _ex).
 * Label smoothing needs each row's sum of logits over the whole vocabulary:
 *   zsum     device [L] float32 out of the forward calls: sum_j z_ij over the
 *            slice's columns (the split sums added in float64, rounded to
 *            float); required when label_smoothing > 0, else may be NULL
 *            (written whenever given). The caller gathers it with m, s, zy.
 *   zsum     device [P][L] float32 in to lce_combine_slices_ex, slice r at
 *            r * L in the order of m, s, zy; required when label_smoothing
 *            > 0, else ignored (may be NULL).
 * The merged loss is the variant's of lce_forward_ex over V_total, and the
 * backward calls give the slice's columns of its G (eps / V_total is the
 * smoothing mass per column, the z-loss factor uses the merged lse). Every
 * process must pass the same opts to all of its calls. Missing zsum or
 * invalid opts return LCE_ERR_INVALID_ARG before anything is queued.
 */
lce_status lce_forward_slice_ex(const void* h, const void* W, lce_dtype dt,
                                const int64_t* labels, int64_t L, int64_t H,
                                int64_t Vs, int64_t v0, int64_t V_total,
                                int64_t ignore_index,
                                const lce_loss_opts* opts, float* m, float* s,
                                float* zy, float* zsum, void* ws,
                                size_t ws_bytes, void* stream);
lce_status lce_combine_slices_ex(const float* m, const float* s,
                                 const float* zy, const float* zsum, int64_t P,
                                 const int64_t* labels, int64_t L,
                                 int64_t V_total, int64_t ignore_index,
                                 const lce_loss_opts* opts, float* loss,
                                 float* lse, void* ws, size_t ws_bytes,
                                 void* stream);
lce_status lce_backward_slice_ex(const void* h, const void* W, lce_dtype dt,
                                 const int64_t* labels, const float* lse,
                                 int64_t L, int64_t H, int64_t Vs, int64_t v0,
                                 int64_t V_total, int64_t ignore_index,
                                 const lce_loss_opts* opts,
                                 const float* dloss, int64_t chunk_rows,
                                 float* dH_part, float* dW, void* ws,
                                 size_t ws_bytes, void* stream);
lce_status lce_forward_slice_exp_ex(const void* h, const void* W,
                                    lce_dtype dt, const int64_t* labels,
                                    int64_t L, int64_t H, int64_t Vs,
                                    int64_t v0, int64_t V_total,
                                    int64_t ignore_index,
                                    const lce_loss_opts* opts, float* m,
                                    float* s, float* zy, float* zsum,
                                    void* ws, size_t ws_bytes, void* stream);
lce_status lce_backward_slice_exp_ex(const void* h, const void* W,
                                     lce_dtype dt, const int64_t* labels,
                                     const float* lse, int64_t L, int64_t H,
                                     int64_t Vs, int64_t v0, int64_t V_total,
                                     int64_t ignore_index,
                                     const lce_loss_opts* opts,
                                     const float* dloss, float* dH_part,
                                     float* dW, void* ws, size_t ws_bytes,
                                     void* stream);

/*
 * Count of rows that take part in the loss: n_valid[0] = #{i : labels[i] !=
 * ignore_index and 0 <= labels[i] < V}. A label that is neither raises
 * LCE_ERR_LABEL_RANGE in the device error word and is not counted, as in
 * lce_forward. This is the N of the mean. When a sequence's rows are split
 * over several processes, as context parallelism splits them ("Training
 * Beyond 1M Tokens", section "One GPU is not enough: split the sequence
 * across many"), the sequence's loss is sum_r N_r loss_r / sum_r N_r over the
 * processes r, not the average of their losses; this call gives each N_r.
 *   labels   device, [L] int64, 8-byte aligned (may be NULL when L = 0)
 *   L        rows, >= 0; V >= 1
 *   n_valid  device, [1] int64 out, 8-byte aligned
 * Queues a memset and (for L > 0) one kernel on `stream`; argument errors
 * return before anything is queued.
 */
lce_status lce_count_valid(const int64_t* labels, int64_t L, int64_t V,
                           int64_t ignore_index, int64_t* n_valid,
                           void* stream);

/*
 * The row-sharded sequence's loss and gradient weights, from each shard's
 * own call. Same source as lce_count_valid; the TRL PR #6845 page ("TRL:
 * document 1M-token training and add a context-parallelism example"),
 * table "Assumptions", lists an evaluation loss that comes out scaled by
 * the number of shards, the kind of mistake a single global N prevents.
 * With shard r's mean loss loss_r over N_r valid rows (lce_forward or
 * lce_forward_backward on its rows, N_r from lce_count_valid):
 *   lce_shard_sums:     sums[0] = N_r loss_r, sums[1] = N_r   (float64)
 *   (the caller sums `sums` over the shards, e.g. one all-reduce)
 *   lce_combine_shards: loss   = S / N                  (S, N the summed pair)
 *                       weight = dloss N_r / N          (dloss NULL: 1)
 *                       both 0 when N = 0
 * Shard r's gradients from the call on its rows (those of its own mean
 * loss) times weight are its share of the sequence's gradients: dH stays on
 * the shard, dW is the sum over the shards (lce_scale_gradients then one
 * all-reduce).
 *   loss_local  device, [1] float32;  n_local device, [1] int64
 *   sums        device, [2] float64 (out of lce_shard_sums, in of
 *               lce_combine_shards), 8-byte aligned
 *   dloss       device, [1] float32 or NULL; loss, weight device [1] float32
 * Each queues one single-thread kernel on `stream`; argument errors return
 * before anything is queued.
 */
lce_status lce_shard_sums(const float* loss_local, const int64_t* n_local,
                          double* sums, void* stream);
lce_status lce_combine_shards(const double* sums, const int64_t* n_local,
                              const float* dloss, float* loss, float* weight,
                              void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device. Returns LCE_ERR_TIMEOUT or LCE_ERR_LABEL_RANGE if a kernel
 * raised one since the last call (timeout first), LCE_ERR_CUDA if the
 * synchronisation failed, else LCE_OK. The word is shared by all streams of
 * the device.
 */
lce_status lce_get_error(void* stream);

/* Human-readable name of a status. Static storage; never NULL. */
const char* lce_status_string(lce_status s);

/* Text of the last CUDA error the library saw on this thread ("" if none). */
const char* lce_last_cuda_error(void);

/*
 * Test hook for the tensor-core building block: D = A B in fp32.
 * No counterpart on the pages; it exposes the contraction kernel alone so
 * that every operand layout can be checked against a plain matmul.
 *   A device bf16: a_mn = 0 -> [M][K] (K-major), a_mn = 1 -> [K][M]
 *   B device bf16: b_mn = 0 -> [N][K] (K-major), b_mn = 1 -> [K][N]
 *   D device fp32 [M][N]; N % 8 == 0; the contiguous dimension of A and B
 *   must be a multiple of 8.
 */
lce_status lce_test_gemm(const void* A, const void* B, float* D, int64_t M,
                         int64_t N, int64_t K, int a_mn, int b_mn,
                         void* stream);

/*
 * Test hook for failure detection: one kernel waits on a barrier that
 * nothing signals, gives up after timeout_ns and raises the timeout bit, so
 * the next lce_get_error returns LCE_ERR_TIMEOUT. No counterpart on the
 * pages. The GPU context stays usable.
 */
lce_status lce_test_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Forward for callers that cannot allocate device memory. No counterpart on
 * the pages: it exists for callers that have no way to provide
 * lce_forward's workspace, such as an embedding runtime that owns all device
 * memory and hands out only the tensors themselves, code that must not
 * allocate after start-up (a frozen memory arena, or a latency-critical loop
 * where cudaMalloc's implicit device synchronisation is not allowed), or a
 * plain C host with no device allocator of its own. It computes exactly what lce_forward
 * computes (bf16 inputs only), taking its scratch from a fixed 16 MiB
 * array inside the library instead of a caller workspace; every GPU that
 * loads the library holds that array until the process exits.
 *   h, W, labels, loss, lse, stream: as for lce_forward (dt = LCE_BF16)
 *   L must be <= 131072 rows; larger L returns LCE_ERR_WORKSPACE (see
 *   lce_last_cuda_error) without queuing anything.
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * All calls share the one array and it keeps the last call's contents, so
 * calls whose work overlaps on the GPU (two streams, or concurrent graph
 * replays) race and give wrong results; order them on one stream.
 * It runs the single-CTA contraction without wave pacing, and at most as
 * many column splits as the array holds at this L (15 at L = 131072), so
 * it is somewhat slower than lce_forward: 96.3 against 88.9 ms at
 * L = 131072, H = 4096, V = 151936 on a GB300.
 */
lce_status lce_forward_static(const void* h, const void* W,
                              const int64_t* labels, int64_t L, int64_t H,
                              int64_t V, int64_t ignore_index, float* loss,
                              float* lse, void* stream);

/*
 * Sequence-tiled gated MLP. Source: "Training Beyond 1M Tokens", section
 * "One GPU is not enough: split the sequence across many": one MLP line of
 * the model is down_proj(act_fn(gate_proj(x)) * up_proj(x)), and its four
 * L x I intermediates are what fills the card at long sequence length. With
 * act_fn = SiLU (the Qwen3 models' activation):
 *   y = (silu(x Wg^T) * (x Wu^T)) Wd^T
 * computed over row chunks, so the intermediates exist only for one chunk
 * (workspace: 10 * chunk_rows * I bytes). The backward recomputes g, u and
 * a per chunk.
 *   x   device bf16 [L][H];  Wg, Wu device bf16 [I][H];  Wd device bf16 [H][I]
 *   y   device bf16 [L][H] out;  dy device bf16 [L][H]
 *   dx  device bf16 [L][H] out;  dWg, dWu fp32 [I][H] out;  dWd fp32 [H][I] out
 *   dx, dWd and the pair (dWg, dWu) may each be NULL, and that gradient's
 *   contraction is skipped (frozen weights: dx alone); not all of them,
 *   and dWg, dWu both or neither. The others keep their bits.
 *   H % 8 == 0, I % 64 == 0; chunk_rows 0 = the library's default.
 * The gate and up projections run as one tensor-core contraction (each
 * 256-row B tile is 128 rows of Wg and the same 128 rows of Wu) whose
 * epilogue writes silu(g) * u; the backward's da = dy Wd contraction writes
 * dg = da u silu'(g) and du = da silu(g); dx = [dg | du] [Wg ; Wu] is one
 * K = 2I contraction; weight gradients accumulate in fp32 in chunk order.
 */
size_t lce_mlp_workspace_size(int64_t L, int64_t H, int64_t I,
                              int64_t chunk_rows);
lce_status lce_mlp_forward(const void* x, const void* Wg, const void* Wu,
                           const void* Wd, int64_t L, int64_t H, int64_t I,
                           int64_t chunk_rows, void* y, void* ws,
                           size_t ws_bytes, void* stream);
lce_status lce_mlp_backward(const void* x, const void* Wg, const void* Wu,
                            const void* Wd, const void* dy, int64_t L,
                            int64_t H, int64_t I, int64_t chunk_rows,
                            void* dx, float* dWg, float* dWu, float* dWd,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Selects how the tensor-core contractions run, for the whole process:
 * enable = 1: on CTA pairs (a cluster of two SMs issues tcgen05.mma with
 * cta_group::2 on 256 x 256 tiles, each SM staging half of each operand);
 * enable = 0: one CTA per 128 x 256 tile. Both give the same results up to
 * fp32 summation order. The environment variable LCE_CTA_PAIR=0/1 sets the
 * initial choice. lce_get_cta_pair returns the current one. No counterpart
 * on the pages. Returns LCE_ERR_INVALID_ARG for other values.
 */
lce_status lce_set_cta_pair(int enable);
int lce_get_cta_pair(void);

/*
 * Wave pacing of the persistent tensor-core contractions, for the whole
 * process: enable = 1 (the default) keeps the CTAs that read the same
 * operand panels within about one output tile of each other, so a panel
 * is fetched from DRAM once per wave of tiles instead of once per CTA that
 * drifted out of L2's reach (a bounded wait on a counter in the workspace
 * before each tile; a wait that runs out goes on, so results never depend
 * on it). enable = 0: every CTA runs free. Results are bit-identical either
 * way. LCE_WAVE_SYNC=0/1 sets the initial choice. No counterpart on the
 * pages. Returns LCE_ERR_INVALID_ARG for other values.
 */
lce_status lce_set_wave_sync(int enable);
int lce_get_wave_sync(void);

/*
 * Per-kernel timing of this library's own launches, for benchmarks. No
 * counterpart on the pages. Between lce_profile_start() and
 * lce_profile_stop(), every kernel the calling thread launches through this
 * library is bracketed by two CUDA events on its stream (a few microseconds
 * per launch). lce_profile_stop waits for those events and fills
 * stats[LCE_KERNEL_KINDS]: per kernel kind, the number of launches, the sum
 * of their event-measured durations, and their algorithmic flops (2 M N K
 * per tensor-core contraction, 0 for the other kernels). Host-side state
 * only; events are created on first use and reused.
 */
#define LCE_KERNEL_KINDS 22
enum {
  LCE_K_COUNT_VALID = 0,
  LCE_K_GEMM_LSE = 1,
  LCE_K_LSE_COMBINE = 2,
  LCE_K_LOSS_FINALIZE = 3,
  LCE_K_F32_TO_BF16 = 4,
  LCE_K_GEMM_GRAD = 5,
  LCE_K_GEMM_DH = 6,
  LCE_K_GEMM_DW = 7,
  LCE_K_TEST_GEMM = 8,
  LCE_K_WAIT_PROBE = 9,
  LCE_K_GEMM_FUSED = 10,
  LCE_K_GRAD_FROM_EXP = 11,
  LCE_K_SCALE_GRADS = 12,
  LCE_K_MLP_GATE_UP = 13,
  LCE_K_MLP_DOWN = 14,
  LCE_K_MLP_DA = 15,
  LCE_K_MLP_DX = 16,
  LCE_K_MLP_DWD = 17,
  LCE_K_MLP_DWGU = 18,
  LCE_K_SLICE_STATS = 19,
  LCE_K_COMBINE_SLICES = 20,
  LCE_K_SHARD_COMBINE = 21
};

typedef struct {
  const char* name; /* static string */
  int64_t launches;
  double total_ms;
  double flops;
} lce_kernel_stat;

lce_status lce_profile_start(void);
lce_status lce_profile_stop(lce_kernel_stat* stats);

#ifdef __cplusplus
}
#endif

#endif /* LCE_H_ */
