/*
 * rnn.h -- C-ABI of librnn: stacked LSTM / GRU / simple-RNN (tanh or ReLU) forward and
 * backward-through-time on one NVIDIA GB300 (sm_103a).
 *
 * The method follows "Optimizing Performance of Recurrent Neural Networks on
 * GPUs" (Appleyard, Kocisky, Blunsom; review page, section "제안 방법"):
 *   - the G gate matrices of a cell are stacked into one matrix so that each
 *     product is one large GEMM (LSTM G=4, GRU G=3, simple RNN G=1);
 *   - the input projection of all timesteps is independent of the recurrence
 *     and runs as one GEMM ahead of it;
 *   - forward and backward passes of consecutive layers overlap (a wavefront:
 *     layer l+1 runs behind layer l);
 *   - the weight update is one GEMM over all timesteps, the bias update a
 *     cheap reduction.
 * From "Persistent RNNs: Stashing Recurrent Weights On-Chip" (Diamos et al.,
 * citing snippets on its page): a small-batch recurrence keeps its recurrent
 * weights on-chip across timesteps and runs every timestep in one launch.
 * The pages print no equations, layouts or API; the cells are the textbook
 * ones (see each call) and the interface below is this library's own.
 *
 * Conventions for every call
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library never allocates device memory and keeps no pointer after a call
 *     returns.  The handle is a host object holding the shape and the
 *     library's launch plan.
 *   - Calls are asynchronous on `stream`; they only enqueue work.  Errors that
 *     the host can see (arguments, launch failures) are returned at once.
 *     A bounded device-side wait that gave up is recorded in the workspace
 *     and reported by rnn_sync_status().
 *   - Element types: in RNN_MODE_BF16, x, y, h0, hT, dy, dhT, dx, dh0 and the
 *     user weights are bfloat16; in RNN_MODE_FP32 they are float.  Cell
 *     states c0, cT, dcT, dc0 and the weight gradient dw are always float.
 *   - Layouts are row-major and time-major:
 *       x[T][B][input], y/dy[T][B][hidden], dx[T][B][input],
 *       h0/c0/hT/cT/dhT/dcT/dh0/dc0[layers][B][hidden].
 *   - User weight layout (same element order as torch.nn.LSTM/GRU/RNN
 *     parameters), per layer l in order:
 *       W_x[G*hidden][I_l], W_h[G*hidden][hidden], b_x[G*hidden], b_h[G*hidden]
 *     with I_0 = input, I_l = hidden for l >= 1, and gate blocks ordered
 *     LSTM (i, f, g, o), GRU (r, z, n), RNN (one block).  dw has the same
 *     layout in float.
 *   - Bidirectional stacks (RNN_FLAG_BIDIRECTIONAL; D = 2, else D = 1): each
 *     layer has a forward and a reverse direction, the reverse one running
 *     from t = T-1 down to 0 from its own initial state.  Weights come per
 *     (layer, direction) v = l*D + d in that order (torch's "_reverse"
 *     parameters after each layer's own), with I_l = D*hidden for l >= 1;
 *     y/dy are [T][B][D*hidden] with y[t] = [h_forward(t), h_reverse(t)];
 *     the state arrays are [layers*D][B][hidden] indexed by v, and hT of the
 *     reverse direction is its state after t = 0.  With rnn_set_lengths()
 *     the reverse direction of each sequence starts at its own last step
 *     from its h0.  Small batches run each direction as one persistent launch.
 *   - Pointers must be 16-byte aligned.  Shapes: in RNN_MODE_BF16 hidden must
 *     be a multiple of 64 and input of 8; in RNN_MODE_FP32 hidden a multiple
 *     of 32 and input of 4 (RNN_ERR_UNSUPPORTED otherwise).
 *   - Return value: RNN_OK (0) or a negative RNN_ERR_* code; rnn_strerror()
 *     names it.  No C++ exception crosses this interface.
 */
#ifndef RNN_H
#define RNN_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define RNN_API __attribute__((visibility("default")))
#else
#define RNN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RNN_LSTM = 0, RNN_GRU = 1, RNN_TANH = 2, RNN_RELU = 3 } rnn_cell_t;
typedef enum { RNN_MODE_FP32 = 0, RNN_MODE_BF16 = 1 } rnn_mode_t;

enum {
  RNN_OK = 0,
  RNN_ERR_INVALID_ARG = -1, /* null handle/pointer, bad size, misaligned buffer */
  RNN_ERR_UNSUPPORTED = -2, /* shape or mode the library does not handle */
  RNN_ERR_LAUNCH = -3,      /* kernel could not be launched (e.g. co-residency) */
  RNN_ERR_CUDA = -4,        /* a CUDA runtime call failed */
  RNN_ERR_TIMEOUT = -5,     /* a bounded device-side wait gave up */
  RNN_ERR_NOMEM = -6        /* host allocation for the handle failed */
};

/* rnn_desc_t.flags */
#define RNN_FLAG_NO_WAVEFRONT 0x1u      /* run layers (and the two directions of a bidirectional layer)
                                           one after another (no overlap) */
#define RNN_FLAG_FORCE_STREAMING 0x2u   /* never use the persistent recurrence */
#define RNN_FLAG_FORCE_PERSISTENT 0x4u  /* use the persistent recurrence or fail */
#define RNN_FLAG_PROFILE 0x8u           /* record per-kernel CUDA-event timings */
#define RNN_FLAG_NO_PAIR 0x20u          /* keep every product on single-CTA 128-row tiles */
#define RNN_FLAG_NO_GRAPH 0x40u         /* enqueue kernels directly; by default a call whose pointers were
                                           seen before replays a cached CUDA graph of its launches */
#define RNN_FLAG_NO_PDL 0x80u          /* launch every kernel after the previous one on its stream has
                                           finished; by default, where one stream carries the call's
                                           launches (one layer, or RNN_FLAG_NO_WAVEFRONT), the tensor-core
                                           kernels start while their predecessor drains (programmatic
                                           dependent launch) and load the packed weights before they wait
                                           on it; the layer wavefront's streams launch without it */
#define RNN_FLAG_NO_TRANSPOSED 0x200u   /* keep the recurrent steps in the h W_h^T orientation */
#define RNN_FLAG_FORCE_TRANSPOSED 0x400u /* take the recurrent steps as W_h h^T (bf16 LSTM / simple RNN,
                                            B <= 256, H % 32 == 0) or fail; by default chosen where it
                                            measured faster (LSTM: H >= 2048, or H >= 1024 and B >= 64,
                                            or H >= 256 and 64 <= B <= 128; simple RNN: H >= 2048) */
#define RNN_FLAG_NO_FUSED_POINT 0x800u  /* transposed LSTM steps: run the pointwise BPTT step as its own
                                           kernel after each product instead of inside its epilogue */
#define RNN_FLAG_NO_PERSIST_CLUSTER 0x1000u /* persistent recurrence: hand h_t over through per-step
                                               arrival counters and L2 reads instead of tagged words
                                               gathered per thread-block cluster */
#define RNN_FLAG_PERSIST_CLUSTER_SYNC 0x8000u /* persistent recurrence, cluster hand-off: end each step with a
                                                barrier across the cluster after the gathered h_{t-1} is scattered
                                                to every CTA; by default the scatter uses asynchronous stores whose
                                                bytes each CTA counts on its own mbarrier, with no cluster-wide
                                                barrier per step */
#define RNN_FLAG_BIDIRECTIONAL 0x2000u /* every layer gets a second direction that runs time backwards
                                          with its own weights (see the layouts below) */
#define RNN_FLAG_FP8_STASH 0x4000u /* bf16 inference: the persistent recurrence keeps W_h on chip as e4m3
                                      (fp8) with one float scale per gate row (half the bf16 footprint), which
                                      lets LSTM and GRU layers up to hidden 2048 and simple RNNs up to 4096
                                      with B <= 8 keep their recurrent weights on chip.  A deliberate
                                      approximation (3 mantissa bits per weight): the forward then computes
                                      with W_h' = e4m3(W_h / s) * s.  Training calls (with a reserve) keep the
                                      bf16 path.  rnn_get_sizes includes the stash in the packed size. */
#define RNN_FLAG_NO_STACK 0x10000u /* bf16, one direction, up to 64 sequences: run the forward recurrence as
                                      step launches (with the layer wavefront) instead of the persistent
                                      stacked recurrence (up to 4 layers per launch, each layer's
                                      [W_x | W_h] rows resident in tensor memory, layer l+1 starting step t
                                      as soon as layer l has finished it) */
#define RNN_FLAG_NO_STACK_BWD 0x40000u /* run the backward recurrence as step launches even where the persistent
                                          stacked backward (the transposed products of up to 4 layers per
                                          launch, up to 64 sequences) fits; RNN_FLAG_NO_STACK turns off both */
#define RNN_FLAG_FORCE_STACK 0x20000u /* use the persistent stacked forward recurrence (also for B <= 8 where
                                         the planner would take the single-layer persistent one) or fail */
#define RNN_FLAG_SLIM_STEP 0x80000u /* bf16 LSTM, transposed steps, more than 128 sequences: run the forward
                                       steps on a kernel with three pipeline stages and one tensor-memory
                                       accumulator (97.5 KB of shared memory, 256 TMEM columns), so that a
                                       CTA of another layer's step can share each SM and stream its weights
                                       while this one runs its epilogue */
#define RNN_FLAG_STEP_CHUNKS 0x100000u /* bf16 LSTM training forward, transposed steps, one direction, fixed
                                        lengths, batch a multiple of 32: run the steps of each chunk after the
                                        first step as one cooperative launch in which each CTA pair loads
                                        h_{t-1} once every pair has stored it (bounded waits; a timeout
                                        reported as RNN_ERR_TIMEOUT); ignored where a step's tiles
                                        outnumber the SM pairs */
#define RNN_FLAG_TEST_SKIP_PUBLISH 0x100u /* test hook: in the persistent recurrences one CTA never
                                             publishes its first step, so the others' bounded waits
                                             give up and rnn_sync_status reports RNN_ERR_TIMEOUT */

typedef struct {
  int cell;             /* rnn_cell_t */
  int layers;           /* L >= 1 */
  int T;                /* timesteps >= 1 */
  int B;                /* batch >= 1 */
  int input;            /* input size of layer 0 */
  int hidden;           /* hidden size H */
  int mode;             /* rnn_mode_t */
  unsigned flags;       /* RNN_FLAG_* */
  long long timeout_ns; /* bound on every device-side wait; <= 0 selects 2 s */
  int chunk;            /* wavefront chunk in timesteps; <= 0 selects automatically */
} rnn_desc_t;

typedef struct rnn_s* rnn_handle_t;

/* Create a handle for one shape.  Validates the descriptor
 * (RNN_ERR_INVALID_ARG / RNN_ERR_UNSUPPORTED) and chooses the launch plan
 * (persistent vs streaming recurrence, wavefront chunk, GEMM tiles) for the
 * current device.  *out receives the handle (host memory, freed by
 * rnn_destroy). */
RNN_API int rnn_create(const rnn_desc_t* desc, rnn_handle_t* out);
RNN_API int rnn_destroy(rnn_handle_t h);

/* Byte sizes of the caller-owned buffers: the user weight vector, the packed
 * weight buffer, the reserve (training state kept from rnn_fwd for the
 * backward calls) and the workspace (scratch for any call).  Any pointer may
 * be NULL. */
RNN_API int rnn_get_sizes(rnn_handle_t h, size_t* user_weight_bytes, size_t* packed_weight_bytes,
                  size_t* reserve_bytes, size_t* workspace_bytes);

/* Weight pack: converts user-layout weights into the packed layout every
 * kernel reads (gate rows interleaved in blocks so that one output tile holds
 * all gates of the same hidden units; biases folded and widened to float).
 * Run once per weight update.  w_user: user layout in the mode's type. */
RNN_API int rnn_pack_weights(rnn_handle_t h, const void* w_user, void* w_packed, cudaStream_t stream);

/* Variable-length sequences (packed-sequence semantics) for later calls on
 * this handle: lens[B] on the host, non-increasing (the batch sorted longest
 * first), 1 <= lens[b] <= T; NULL = every sequence runs all T steps.
 * Sequence b runs steps 0 .. lens[b]-1: y is 0 at its later steps, hT / cT
 * receive its state after its own last step, its dy at later steps is
 * ignored, dhT / dcT enter at its last step, and dx is 0 at later steps.
 * Padding in x past a sequence's end must be finite (it meets zero gate
 * gradients in the weight-gradient product).  At each step only the
 * sequences still running are computed.  A handle that had planned the
 * persistent recurrence switches to per-step launches; cached launch graphs
 * are dropped (after a device-wide synchronize, so call it between steps,
 * not while this handle's work is being captured).  Bidirectional stacks:
 * the reverse direction of sequence b starts at step lens[b]-1 from its h0.
 * Returns RNN_ERR_INVALID_ARG for unsorted or out-of-range lengths (nothing
 * changes then).  A handle is not safe to use from several host threads at
 * once. */
RNN_API int rnn_set_lengths(rnn_handle_t h, const int* lens);

/* Forward pass over all layers and timesteps.  Per layer l and step t:
 *   LSTM: a = W_x in_t + b_x + W_h h_{t-1} + b_h; i,f,o = sigmoid, g = tanh;
 *         c_t = f*c_{t-1} + i*g;  h_t = o*tanh(c_t)
 *   GRU:  r,z = sigmoid(W_x in + b_x + W_h h + b_h) (their gate blocks);
 *         n = tanh(W_xn in + b_xn + r*(W_hn h_{t-1} + b_hn));
 *         h_t = (1-z)*n + z*h_{t-1}
 *   RNN:  h_t = tanh(W_x in_t + b_x + W_h h_{t-1} + b_h)
 *   ReLU RNN: h_t = max(0, W_x in_t + b_x + W_h h_{t-1} + b_h) (slope 0 at the kink).
 *         The pages name the simple RNN without its activation; tanh is the
 *         named target, ReLU the other common choice for the cell.
 * with in_t = x_t for layer 0 and h^{l-1}_t above it.  y_t = h^{L-1}_t.
 * h0/c0 NULL mean zero state; hT/cT NULL are not written; c-arguments are
 * ignored for GRU and RNN.  reserve == NULL runs inference; otherwise the
 * reserve receives what rnn_bwd_data needs.  ws: workspace of
 * rnn_get_sizes() bytes. */
RNN_API int rnn_fwd(rnn_handle_t h, const void* x, const void* h0, const float* c0, const void* w_packed,
            void* y, void* hT, float* cT, void* reserve, void* ws, cudaStream_t stream);

/* Backward pass through time for the data gradients: the exact gradient of
 * sum(y*dy) + sum(hT*dhT) + sum(cT*dcT) with respect to x, h0 and c0,
 * computed top layer first in reverse time.  It also leaves the gate
 * gradients in the reserve for rnn_bwd_weights.  Must follow rnn_fwd with the
 * same reserve.  dhT/dcT NULL count as zero; dx/dh0/dc0 NULL are not
 * written. */
RNN_API int rnn_bwd_data(rnn_handle_t h, const void* dy, const void* dhT, const float* dcT,
                 const void* w_packed, const void* h0, const float* c0, void* dx, void* dh0,
                 float* dc0, void* reserve, void* ws, cudaStream_t stream);

/* Weight gradients, one GEMM per layer and weight matrix over all T*B rows:
 *   dW_x = sum_t dGx_t^T in_t,  dW_h = sum_t dGh_t^T h_{t-1},
 *   db_x = sum dGx, db_h = sum dGh
 * written in the user layout as float.  accumulate != 0 adds to dw instead
 * of overwriting it.  Must follow rnn_bwd_data with the same reserve. */
RNN_API int rnn_bwd_weights(rnn_handle_t h, const void* x, const void* h0, const void* reserve, float* dw,
                    int accumulate, void* ws, cudaStream_t stream);

/* Synchronizes `stream`, then reads and clears the device error word in the
 * workspace: RNN_OK, RNN_ERR_TIMEOUT if a bounded device wait gave up in any
 * call since the last check, or RNN_ERR_LAUNCH if the persistent recurrence
 * found itself launched in clusters of another size than planned (it then
 * computes nothing). */
RNN_API int rnn_sync_status(rnn_handle_t h, void* ws, cudaStream_t stream);

RNN_API const char* rnn_strerror(int code);

/* Plan introspection: writes a short text description of the chosen launch
 * plan (recurrence kind, chunk, tiles) into buf (NUL-terminated). */
RNN_API int rnn_describe(rnn_handle_t h, char* buf, size_t len);

/* Number of kernels this library has launched since it was loaded. */
RNN_API unsigned long long rnn_launch_count(void);

/* With RNN_FLAG_PROFILE set, per-kernel-class CUDA-event timings of the calls
 * made since the last reset.  Synchronizes the device.  For class index k
 * (0 <= k < *n_classes) fills name (up to 32 chars), launches and total
 * milliseconds; returns RNN_ERR_INVALID_ARG for k out of range.  reset != 0
 * clears the records afterwards. */
RNN_API int rnn_profile_query(rnn_handle_t h, int k, char* name, int* n_classes,
                      unsigned long long* launches, double* total_ms, int reset);

/* ------------------------------------------------------------------------
 * Building block exposed for tests: the tcgen05 GEMM engine the input
 * projection, the data-gradient and the weight-gradient products run on.
 *   D[m][n] = sum_k A(m,k) * B(n,k)  (+ bias[n]) (+ D[m][n] if accumulate)
 * A(m,k) = A[m*lda + k] when a_mn_major == 0, else A[k*lda + m]; B likewise.
 * A, B bfloat16 on the device; D, bias float.  bias may be NULL.
 * ---------------------------------------------------------------------- */
RNN_API int rnn_gemm_bf16(int M, int N, int K, const void* A, long long lda, int a_mn_major,
                  const void* B, long long ldb, int b_mn_major, float* D, long long ldd,
                  const float* bias, int accumulate, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Building block exposed for tests: the per-row e4m3 quantisation of the
 * fp8 stash (RNN_FLAG_FP8_STASH).  w: bf16 [rows][cols] on the device;
 * scale[r] = max_k |w[r][k]| / 448 (1 for an all-zero row) and
 * q[r][k] = e4m3(w[r][k] / scale[r]), round to nearest even.
 * ---------------------------------------------------------------------- */
RNN_API int rnn_quantize_e4m3_rows(int rows, int cols, const void* w, void* q, float* scale, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Bias gradients with no workspace and no allocation.  The paper has no
 * counterpart; this exists for callers that cannot allocate device memory
 * when they need the result: for example a host framework that hands a
 * plugin fixed input/output buffers only and forbids cudaMalloc after
 * start-up (it synchronizes the device and can fail under memory pressure),
 * so there is no room for the workspace rnn_bwd_weights takes.
 *
 * Computes db_x and db_h of every layer (and, in bidirectional stacks, of
 * both directions of every layer) from the gate gradients that
 * rnn_bwd_data left in `reserve`, and writes them into `dw` (user layout,
 * float) at the same places rnn_bwd_weights does; dW_x and dW_h in `dw` are
 * not touched.  accumulate != 0 adds instead of overwriting.
 *
 * Scratch: a fixed array of RNN_BIAS_STATIC_FLOATS floats (4 MiB) inside
 * the library, held by every GPU that loads it until the process exits.
 * G*hidden must not exceed RNN_BIAS_STATIC_FLOATS (RNN_ERR_UNSUPPORTED).
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  All calls
 * share the one array: calls that overlap on the GPU (other streams, other
 * handles) race and must be ordered by the caller.
 * ---------------------------------------------------------------------- */
#define RNN_BIAS_STATIC_FLOATS (1 << 20)
RNN_API int rnn_bias_grad_static(rnn_handle_t h, const void* reserve, float* dw, int accumulate,
                                 cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* RNN_H */
