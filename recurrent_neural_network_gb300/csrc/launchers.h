// launchers.h -- host-side entry points of the kernel translation units, used
// by the C-ABI layer (api.cu).  Plain pointers and sizes only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rnn {

// One GEMM operand: element (mn, k) sits at ptr[mn*ld + k] (K-major) or
// ptr[k*ld + mn] (MN-major).  Elements outside [0,mn_ext) x [0,k_ext) are zero.
struct Operand {
  const void* ptr;
  long long ld;
  int mn_major;
  int mn_ext, k_ext;
  // 1: no kernel that may still be running writes this operand (packed
  // weights), so a dependent launch may start loading it before it waits
  int is_static = 0;
};

struct Profiler;  // defined in api.cu

// Launch context: stream, device error word, wait bound, SM count, and the
// profiling hook (null = off) with the kernel-class name to file timings under.
struct Launch {
  cudaStream_t stream;
  int* err;
  uint64_t limit_ns;
  int num_sms;
  Profiler* prof;
  const char* name;
  int pair = 1;  // products with more than 128 rows may run on CTA pairs (256-row tiles)
  int pdl = 0;   // launch as a programmatic dependent of the previous kernel on the stream
};

// profiling / counting hooks (api.cu)
void launch_begin(const Launch& L);
void launch_end(const Launch& L, int n_kernels = 1);

// Packed -> user row mapping of the weight-gradient products.
struct Remap {
  int on, G, u, H;
};

// ---------------------------------------------------------------- gemm.cu
// Device-to-device copies (1-D, and rows of `width` bytes between pitched
// buffers) and zero fills as kernels on the stream (any alignment; 16-byte
// vectors where every address, pitch and size allows).
int dev_copy(const Launch& L, void* dst, const void* src, size_t bytes);
int dev_copy2d(const Launch& L, void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t rows);
int dev_zero(const Launch& L, void* dst, size_t bytes);
// Up to kMaxDevOps copies (src non-null) and zero fills (src null) in one launch.
struct DevOp {
  void* dst;
  const void* src;
  size_t bytes;
};
constexpr int kMaxDevOps = 16;
int dev_batch(const Launch& L, const DevOp* ops, int n);
// D[m][n] = sum_k A(m,k) B(n,k) (+ bias[n]) (+ D) with float output.
// mode 1: bf16 operands on tcgen05; mode 0: fp32 operands on FFMA.
int gemm_f32(const Launch& L, int mode, const Operand& A, const Operand& B, int M, int N, int K, float* D,
             long long ldd, const float* bias, int accumulate, const Remap& remap, int max_ctas);
// same with storage-type output (bf16 in mode 1, float in mode 0)
int gemm_store(const Launch& L, int mode, const Operand& A, const Operand& B, int M, int N, int K, void* D,
               long long ldd, int max_ctas);

// user -> packed weights for one layer
int pack_layer(const Launch& L, int mode, int cell, int H, int In, int u, const void* wx, const void* wh,
               const void* bx, const void* bh, void* pwx, void* pwh, float* pbias, float* pbias_hn);

// column sums over `rows` rows of the gate-gradient matrices into user-layout
// bias gradients (gate blocks of H).  dgh may equal dgx.  part: scratch of
// slices * G*H floats.
int bias_grad(const Launch& L, int mode, int cell, int H, int u, long long rows, const void* dgx, const void* dgh,
              float* dbx, float* dbh, int accumulate, float* part, int slices);
// dst[i] = src[i] rounded to bf16 (n a multiple of 4; both 16-byte aligned)
int cast_bf16(const Launch& L, const float* src, void* dst, size_t n);
// Per-row e4m3 quantisation of a bf16 matrix w[rows][cols]: scale[r] =
// max_k |w[r][k]| / 448 (1 for an all-zero row) and q[r][k] = e4m3(w / scale)
// rounded to nearest even (|w / scale| <= 448 by construction).
int quant_rows_e4m3(const Launch& L, const void* w, int rows, int cols, uint8_t* q, float* scale);

// ---------------------------------------------------------------- step_fwd.cu
struct FwdStepArgs {
  int B, H, u;
  float* P;
  int write_gates;
  const float* bias_hn;
  const float* c_prev;
  float* c_out;
  const void* h_prev;
  void* h_out;
  void* y;
  void* hT;
  float* cT;
  float* hn_out;
  int slim = 0;  // transposed LSTM steps over more than 128 sequences: the shared-SM kernel
  // transposed LSTM steps, several in one launch: `steps` consecutive steps
  // whose P, c, h_prev / h_out and y follow one another B rows apart (c_prev
  // of step s is c_out of step s-1); hT / cT written by step hT_step (none
  // when out of range); step_cnt: `steps` zeroed arrival counters
  int steps = 1, hT_step = -1;
  unsigned int* step_cnt = nullptr;
};
// one forward timestep of one layer: A = h_{t-1} [B][H], B = packed W_h [G*H][H]
int fwd_step(const Launch& L, int mode, int cell, const Operand& A, const Operand& Bw, const FwdStepArgs& a);
// the same step transposed (bf16, LSTM / tanh RNN, packing unit 1):
// A = packed W_h [G*H][H], B = h_{t-1} [B][H]; tiles of 256 gate rows x the batch
int fwd_step_t(const Launch& L, int cell, const Operand& Wh, const Operand& Hp, const FwdStepArgs& a);

// ---------------------------------------------------------------- step_bwd.cu
struct BwdStepArgs {
  int B, H, u;
  const float* gates;
  const float* c_s;
  const float* c_sm1;
  const float* hn_s;
  const void* h_sm1;
  const void* dy;
  int dy_f32;
  float* carry;
  void* dGx;
  void* dGh;
  int final_;
  void* dh0;
  float* dc0;
  float* part;
  int* counters;
  int cluster_splitk;  // reduce split-K partials inside a thread-block cluster instead of through global memory
};
// one backward timestep: A = dGh_{s+1} [B][G*H], Bw = packed W_h (MN-major view)
int bwd_step(const Launch& L, int mode, int cell, const Operand& A, const Operand& Bw, int bn, int splits,
             const BwdStepArgs& a);
// pointwise-only backward step (the last timestep): dh starts from dh_init
// ([B][H], storage type, null = zero)
int bwd_point(const Launch& L, int mode, int cell, const BwdStepArgs& a, const void* dh_init);
// Transposed backward product (bf16, packing unit 1): A = packed W_h read
// MN-major ([H] x [G*H]), B = dG_{s+1} [B][G*H]; tiles of 128 hidden units x
// the batch, K split `splits` ways inside clusters.  Writes dh (fp32 [B][H]),
// or dh0 (bf16 [B][H]) when final_ (dh0 null: nothing to write).
// pf_*: inputs of the pointwise step that follows, pulled into L2 near the
// end of the product's mainloop (null: none)
// Tiles are 128 units x bn (64, 128 or 256) batch entries; with splits > 1
// the partial sums pass through `part` (fp32, splits * ceil(B/bn)*bn * H).
// fuse non-null (LSTM, bn = 256, 4 splits): the pointwise step runs inside
// the product's epilogue with these arguments (dh is then not written).
struct PointVArgs;
int bwd_dh_t(const Launch& L, const Operand& WhT, const Operand& dG, int B, int H, int G, int bn, int splits,
             float* dh, void* dh0, int final_, float* part, const float* pf_gates = nullptr,
             const float* pf_c_s = nullptr, const float* pf_c_sm1 = nullptr, const PointVArgs* fuse = nullptr);
// the pointwise backward step that follows it (packing unit 1, H % 4 == 0)
struct PointVArgs {
  int B, H;
  const float* dh;      // product part of dh_s, or null
  const void* dh_init;  // bf16 [B][H] used when dh is null, or null = zero
  const void* dy;       // [B][H] gradient from above, float if dy_f32 else bf16, or null
  int dy_f32;
  const float* gates;   // [B][G*H]
  const float* c_s;     // LSTM
  const float* c_sm1;   // LSTM, null = zero
  float* carry;         // LSTM
  float* dc0;           // LSTM, step 0 only: copy of the outgoing carry, or null
  void* dGx;            // bf16 [B][G*H]
};
int bwd_point_v(const Launch& L, int cell, const PointVArgs& a);

// ---------------------------------------------------------------- persist.cu
struct PersistArgs {
  int T, B, H, u_pack, uc;
  const __nv_bfloat16* Wh;  // packed [G*H][H]
  const uint8_t* Wh8;       // fp8 stash: packed [G*H][H] e4m3 bytes (null: bf16 fragments from Wh)
  const float* wscale;      // fp8 stash: scale of each packed row
  const float* P;           // [T][B][G*H] input projection incl. bias
  float* gates_out;         // training: activated gates [T][B][G*H] (may alias P), else null
  const float* bias_hn;     // GRU [H]
  const float* c0;          // LSTM [B][H] or null
  float* c_out;             // LSTM training [T][B][H] or null
  float* hn_out;            // GRU training [T][B][H] or null
  __nv_bfloat16* hseq;      // [T+1][B][H]; slot 0 = h0
  unsigned int* arrive;     // [T] arrival counters, zero before the launch
  int cluster;              // > 0: cluster-exchange hand-off with clusters of this size
  int cluster_sync;         // cluster exchange ended by a barrier across the cluster each step
                            // (0: each CTA waits on its own mbarrier for asynchronous stores)
  uint64_t* hx;             // cluster exchange: [2][B*H/2] tagged words, zero before the launch
  __nv_bfloat16* y;         // [T][B][H] or null
  __nv_bfloat16* hT;        // [B][H] or null
  float* cT;                // [B][H] or null
  int* err;
  uint64_t limit_ns;
  int test_skip_publish;    // test hook: CTA 0 never publishes h_0
  int reverse;              // 1: time runs T-1 .. 0 (P, gates, c, y indexed by time; h(time) at hseq
                            // slot time, the initial state at slot T)
};
// RNN_OK if the persistent recurrence supports (cell, H, B) and all its CTAs
// fit on the device at once; *ctas receives the grid size and *cluster (if
// not null) the largest cluster size (8, 4 or 2) whose clusters all fit at
// once for the cluster-exchange hand-off, 0 if none.  fp8: with the e4m3
// stash of W_h.
int persist_check(int cell, int H, int B, int num_sms, int* ctas, int* cluster = nullptr, bool fp8 = false);
// all T timesteps of one layer in one cooperative launch (bf16 storage only)
int persist_fwd(const Launch& L, int cell, const PersistArgs& a);

// ---------------------------------------------------------------- stack.cu
// Persistent forward recurrence of up to kStackMaxLayers stacked layers in one
// launch (bf16, one direction, 1..64 sequences): each layer's CTAs hold
// blocks of its packed [W_x | W_h] rows on chip, layer l works on step t as
// soon as layer l-1 has finished it (per-layer, per-step arrival counters).
constexpr int kStackMaxLayers = 4;
struct StackLayer {
  const __nv_bfloat16* Wx;  // packed [G*H][In] (layers without P)
  const __nv_bfloat16* Wh;  // packed [G*H][H]
  const float* P;           // [T][B][G*H] input projection incl. bias (the stack's first layer), else null
  const float* bias;        // packed folded bias [G*H] (layers without P)
  const float* bias_hn;     // GRU [H]
  const float* c0;          // LSTM [B][H] or null
  float* gates_out;         // training: activated gates [T][B][G*H] (may alias P), else null
  float* c_out;             // training LSTM [T][B][H], else null
  float* hn_out;            // training GRU [T][B][H], else null
  __nv_bfloat16* hseq;      // [T+1][B][H]; slot 0 = h0, written before the launch
  const __nv_bfloat16* in;  // layers without P: the layer below's h sequence [T+1][B][In] (its output at t in slot t+1)
  __nv_bfloat16* y;         // [T][B][H] or null
  __nv_bfloat16* hT;        // [B][H] or null
  float* cT;                // LSTM [B][H] or null
  int In;                   // input width of a layer without P (must equal H)
  int wait_in;              // 1: the input is produced by the previous layer of this launch
};
struct StackSmem {
  int stages, a, ring, rbuf, smg, smhn, bars;
};
struct StackArgs {
  int T, B, H, u_pack;
  int nl;                   // layers in this launch
  StackLayer lay[kStackMaxLayers];
  unsigned int* cnt;        // [nl][T] arrival counters, zero before the launch
  int* err;
  uint64_t limit_ns;
  int test_skip_publish;    // test hook: CTA 0 never publishes step 0
  // geometry (filled by stack_fwd)
  int cluster;
  int kcl[kStackMaxLayers];  // K chunk width of each layer's CTAs
  int kctl[kStackMaxLayers]; // the first kctl of it in tensor memory, the rest (if any) in shared memory
  int ks[kStackMaxLayers], kcx[kStackMaxLayers], cta0[kStackMaxLayers + 1], ctas[kStackMaxLayers];
  StackSmem sm;
};
// RNN_OK if nl stacked layers of (cell, H, B) run as one stack launch on the
// device (first_p: the first of them reads a precomputed input projection;
// u_pack: the packing unit); *ctas receives the grid size.  num_sms <= 0:
// host-side planning for GB300 without a device query.
// *wide (optional) is set to 1 when some layer needs K chunks wider than
// TMEM holds beside the accumulators (part of its weights in shared memory).
int stack_check(int cell, int H, int B, int nl, int first_p, int u_pack, int num_sms, int* ctas, int* wide = nullptr);
int stack_fwd(const Launch& L, int cell, const StackArgs& a);

// Persistent backward-through-time of up to kStackMaxLayers stacked layers in
// one launch (bf16, one direction, no variable lengths): each CTA owns 128
// hidden units and holds their columns of [W_h^l ; W_x^{l+1}] (one K chunk)
// in tensor memory; layer l works on reverse step s once it has its own
// dGh_{s+1} and the layer above's dGx_s.  lay[0] is the lowest layer.
struct StackBwdLayer {
  const __nv_bfloat16* Wh;        // packed [G*H][H] of this layer
  const __nv_bfloat16* Wx_above;  // packed W_x [G*H][H] of the layer above, null at the top of the stack
  __nv_bfloat16* dgx;             // [T][B][G*H] gate gradients (written)
  __nv_bfloat16* dgh;             // [T][B][G*H] recurrent-side gate gradients (GRU; others: = dgx)
  const __nv_bfloat16* dgx_above; // the layer above's dgx, null at the top of the stack
  const float* gates;             // [T][B][G*H] activated gates
  const float* c;                 // LSTM [T][B][H]
  const float* c0;                // LSTM [B][H] or null
  const float* hn;                // GRU [T][B][H]
  const __nv_bfloat16* hseq;      // GRU: [T+1][B][H] (h_{s-1} in slot s)
  const void* dy;                 // gradient from above [T][B][H]: the user's dy (bf16) at the top of the
                                  // stack, or (dy_f32) a float gradient computed before the launch, or null
  int dy_f32;
  const __nv_bfloat16* dhT;       // [B][H] or null
  const float* dcT;               // LSTM [B][H] or null
  __nv_bfloat16* dh0;             // [B][H] or null
  float* dc0;                     // LSTM [B][H] or null
  int wait_above;                 // 1: the layer above runs in this launch
};
struct StackBwdArgs {
  int T, B, H, u_pack;
  int nl;
  StackBwdLayer lay[kStackMaxLayers];
  unsigned int* cnt;  // [nl][T] arrival counters, zero before the launch
  int* err;
  uint64_t limit_ns;
  int test_skip_publish;
  int budget;  // most CTAs of the launch (from stack_bwd_check)
  // geometry (filled by stack_bwd)
  int cluster;
  int kcl[kStackMaxLayers], ks[kStackMaxLayers], kr[kStackMaxLayers], cta0[kStackMaxLayers + 1],
      ctas[kStackMaxLayers];
  int kctl[kStackMaxLayers];  // the first kctl of each chunk in TMEM, the rest (if any) in shared memory
  StackSmem sm;
};
// RNN_OK if nl stacked layers of (cell, H, B) run their BPTT as one launch
// (has_top: the group's highest layer is the top of the stack, with no layer
// above it); *ctas receives the grid size and *budget the CTA budget to pass
// in StackBwdArgs::budget (the geometry the device can hold).
int stack_bwd_check(int cell, int H, int B, int nl, int has_top, int u_pack, int num_sms, int* ctas, int* budget);
int stack_bwd(const Launch& L, int cell, const StackBwdArgs& a);

}  // namespace rnn
