/*
 * rnn_ref.h -- double-precision CPU oracle for stacked LSTM / GRU / simple-RNN
 * (tanh or ReLU) forward and backward-through-time passes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this code; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no source with the CUDA path.
 *
 * What it computes follows the cells named by "Optimizing Performance of
 * Recurrent Neural Networks on GPUs" (review page, section "제안 방법":
 * LSTM with four gate matrices, GRU with three, simple RNN with one), written
 * out as their textbook definitions because the pages print no equations.
 *
 * Layouts (all row-major, time-major, host memory, double):
 *   x[T][B][I], y[T][B][H], h0/c0/hT/cT/dh0/dc0[L][B][H], dy[T][B][H]
 *   w: per layer l (in order): W_x[G*H][I_l], W_h[G*H][H], b_x[G*H], b_h[G*H]
 *      with I_0 = I, I_l = H for l >= 1, gate blocks LSTM (i,f,g,o),
 *      GRU (r,z,n), RNN tanh / ReLU (single block).
 *   dw: same layout as w.
 * Nullable: h0, c0 (zero state), hT, cT (not written), dhT, dcT (zero),
 *   dx, dh0, dc0 (not written).  c-arguments are ignored for GRU and RNN.
 * Returns 0 on success, -1 on invalid arguments.
 */
#ifndef RNN_REF_H
#define RNN_REF_H
#ifdef __cplusplus
extern "C" {
#endif

enum { RNN_REF_LSTM = 0, RNN_REF_GRU = 1, RNN_REF_TANH = 2, RNN_REF_RELU = 3 };

int rnn_ref_fwd(int cell, int L, int T, int B, int I, int H,
                const double* x, const double* h0, const double* c0, const double* w,
                double* y, double* hT, double* cT);

int rnn_ref_bwd(int cell, int L, int T, int B, int I, int H,
                const double* x, const double* h0, const double* c0, const double* w,
                const double* dy, const double* dhT, const double* dcT,
                double* dx, double* dh0, double* dc0, double* dw);

/* number of OpenMP threads the oracle runs on */
int rnn_ref_threads(void);

/* The same with per-sequence lengths lens[B] (0 <= lens[b] <= T; null = all T):
 * sequence b runs steps 0 .. lens[b]-1, its later outputs are 0 and its state
 * is carried unchanged, so hT / cT are its state after its own last step. */
int rnn_ref_fwd_len(int cell, int L, int T, int B, int I, int H, const int* lens,
                    const double* x, const double* h0, const double* c0, const double* w,
                    double* y, double* hT, double* cT);
int rnn_ref_bwd_len(int cell, int L, int T, int B, int I, int H, const int* lens,
                    const double* x, const double* h0, const double* c0, const double* w,
                    const double* dy, const double* dhT, const double* dcT,
                    double* dx, double* dh0, double* dc0, double* dw);

/* Bidirectional stacks (D = 2; D = 1 is the unidirectional case above).  Each
 * layer l has D sets of weights, v = l*D + d, in that order in w and dw:
 * W_x[G*H][I_l], W_h[G*H][H], b_x[G*H], b_h[G*H] with I_0 = I, I_l = D*H.
 * Direction 1 runs time backwards (from lens[b]-1, or T-1, down to 0, from its
 * own h0).  y[T][B][D*H] holds [h_dir0(t), h_dir1(t)]; h0, c0, hT, cT, dh0,
 * dc0, dhT, dcT are [L*D][B][H] (index v); dy is [T][B][D*H].  hT of
 * direction 1 is its state after time 0. */
int rnn_ref_fwd_dir(int cell, int L, int D, int T, int B, int I, int H, const int* lens,
                    const double* x, const double* h0, const double* c0, const double* w,
                    double* y, double* hT, double* cT);
int rnn_ref_bwd_dir(int cell, int L, int D, int T, int B, int I, int H, const int* lens,
                    const double* x, const double* h0, const double* c0, const double* w,
                    const double* dy, const double* dhT, const double* dcT,
                    double* dx, double* dh0, double* dc0, double* dw);

/* The same, with the on/off decisions of the ReLU cell taken in the precision
 * the device stores h in: decide = 0 (double, as above), 1 (bf16) or 2
 * (fp32): a first forward pass rounds h to that type after every step and
 * records each unit's decision a > 0; or decide = 3: the decisions are given
 * in `on`.  All values are then computed in double with those decisions
 * imposed (h = a where on, 0 where off, slope 1 where on).
 *   on:     [L*D][T][B][H] (by time), nullable unless decide = 3; receives the
 *           decisions taken when decide < 3
 *   preact: [L*D][T][B][H], nullable (forward only); receives the ReLU
 *           pre-activations of the pass that took the decisions
 * Other cells ignore decide, on and preact. */
int rnn_ref_fwd_kp(int cell, int L, int D, int T, int B, int I, int H, const int* lens, int decide,
                   unsigned char* on, double* preact,
                   const double* x, const double* h0, const double* c0, const double* w,
                   double* y, double* hT, double* cT);
int rnn_ref_bwd_kp(int cell, int L, int D, int T, int B, int I, int H, const int* lens, int decide,
                   unsigned char* on,
                   const double* x, const double* h0, const double* c0, const double* w,
                   const double* dy, const double* dhT, const double* dcT,
                   double* dx, double* dh0, double* dc0, double* dw);

#ifdef __cplusplus
}
#endif
#endif
