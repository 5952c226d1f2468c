// api.cu -- the C-ABI of librnn: handle, buffer layouts, launch plan and the
// layer-wavefront scheduler.
//
// Scheduling ("Optimizing Performance of Recurrent Neural Networks on GPUs",
// review page, section "제안 방법": input and recurrent products are
// independent; forward and backward passes of consecutive layers overlap):
//   * layer 0's input projection for all T timesteps is one GEMM;
//   * time is cut into chunks; layer l >= 1 projects its input chunk c as
//     soon as layer l-1 has produced that chunk, then runs the chunk's
//     recurrent steps.  Each layer owns a stream and (layer, chunk) events
//     order the chunks, so layer l+1 works on chunk c while layer l works on
//     chunk c+1 -- the wavefront.  The backward pass runs the same diagram
//     top layer first in reverse time.
//   * small-batch recurrences run all their timesteps in one persistent
//     launch with the recurrent weights held on-chip (see persist.cu).
//   * variable lengths (rnn_set_lengths): with the batch sorted longest
//     first, the sequences running at time t are a prefix of the batch, so
//     every step launch simply gets fewer rows.
//   * bidirectional stacks (fwd_bidir, bwd_bidir, wgrad_bidir): every layer
//     has a second direction that walks time backwards; the two directions
//     of a layer run side by side, layers one after another.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/rnn.h"
#include "launchers.h"

namespace rnn {

// ---------------------------------------------------------------- profiling
struct Profiler {
  struct Rec {
    int cls;
    cudaEvent_t a, b;
    bool graph = false;  // recorded by a captured graph: its events belong to that graph
  };
  bool capturing = false;
  std::vector<Rec> captured;
  std::mutex mu;
  std::vector<std::string> names;
  std::vector<unsigned long long> launches;
  std::vector<double> total_ms;
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;
  Rec open{};

  int cls_of(const char* n) {
    for (size_t i = 0; i < names.size(); ++i)
      if (names[i] == n) return (int)i;
    names.emplace_back(n);
    launches.push_back(0);
    total_ms.push_back(0.0);
    return (int)names.size() - 1;
  }
  cudaEvent_t event() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void settle() {  // requires the device to be idle
    for (auto& r : pending) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
        total_ms[r.cls] += ms;
        launches[r.cls] += 1;
      }
      if (!r.graph) {
        pool.push_back(r.a);
        pool.push_back(r.b);
      }
    }
    pending.clear();
  }
  ~Profiler() {
    for (auto& r : pending) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    for (auto e : pool) cudaEventDestroy(e);
  }
};

static std::atomic<unsigned long long> g_launches{0};

void launch_begin(const Launch& L) {
  if (!L.prof) return;
  Profiler& p = *L.prof;
  std::lock_guard<std::mutex> g(p.mu);
  p.open.cls = p.cls_of(L.name ? L.name : "kernel");
  p.open.graph = p.capturing;
  if (p.capturing) {  // events owned by the graph being captured
    cudaEventCreate(&p.open.a);
    cudaEventCreate(&p.open.b);
  } else {
    p.open.a = p.event();
    p.open.b = p.event();
  }
  cudaEventRecord(p.open.a, L.stream);
}

void launch_end(const Launch& L, int n_kernels) {
  g_launches += (unsigned long long)n_kernels;
  if (!L.prof) return;
  Profiler& p = *L.prof;
  std::lock_guard<std::mutex> g(p.mu);
  cudaEventRecord(p.open.b, L.stream);
  if (p.capturing) p.captured.push_back(p.open);
  else p.pending.push_back(p.open);
}

}  // namespace rnn

using namespace rnn;

// ---------------------------------------------------------------- the handle
struct rnn_s {
  rnn_desc_t d{};
  int G = 0, GH = 0, u = 0, elem = 0;
  int D = 1;  // directions per layer (2: bidirectional); per-(layer, direction) arrays are indexed v = l*D + d
  int num_sms = 152;
  int have_device = 0;
  // plan
  int chunk = 1, nch = 1, wavefront = 0, bwd_bn = 128, bwd_splits = 1;
  int persist = 0, persist_ctas = 0;  // forward recurrence kind: 1 = persistent (one launch per layer)
  int persist_plan = 0;               // the kind the plan chose (variable lengths turn it off)
  int persist_cl = 0;                 // persistent hand-off: cluster size of the tagged-word exchange, 0 = counters
  int persist8 = 0, persist8_cl = 0;  // fp8 stash (RNN_FLAG_FP8_STASH): persistent inference on e4m3 W_h
  int tstep = 0;      // 1: transposed recurrent steps (W_h as the row operand, packing unit 1)
  int slim_step = 0;  // 1: transposed LSTM forward steps on the shared-SM kernel (three stages, one accumulator)
  int step_chunks = 0;  // 1: transposed LSTM training steps of a chunk (after t = 0) in one cooperative launch
  // persistent stacked forward (9..64 sequences): groups of up to
  // kStackMaxLayers layers, each group one launch; stack_plan is the plan's
  // choice, stack what the current lengths allow (variable lengths: off)
  int stack = 0, stack_plan = 0;
  std::vector<std::pair<int, int>> stack_groups;  // (first layer, layers)
  // persistent stacked backward: groups from the top of the stack down
  int stackb = 0, stackb_plan = 0;
  int stackb_rec = 0;  // recurrent-only tops: each group's top layer without the share from above, which a GEMM computes before the group
  std::vector<std::pair<int, int>> stackb_groups;  // (lowest layer, layers), highest group first
  std::vector<int> stackb_budget;                  // CTA budget of each group's geometry
  int bwd_fuse = 0;   // transposed LSTM: the pointwise BPTT step runs inside the product's epilogue
  // variable lengths (rnn_set_lengths): Bt[t] = number of sequences still
  // running at step t (the batch is sorted by non-increasing length, so the
  // running ones are rows 0 .. Bt[t]-1); Bt[T] = 0
  int varlen = 0;
  std::vector<int> Bt;
  uint64_t limit_ns = 2000000000ull;
  // sizes (bytes)
  size_t user_w_bytes = 0, packed_bytes = 0, reserve_bytes = 0, ws_bytes = 0;
  struct PL { size_t wx, wh, bias, bias_hn, wh8, wsc; };
  struct RL { size_t gates, c, hn, hseq, dgx, dgh; };
  struct WL { size_t P, hseq, c2, dyab, carry, part, ctr, dh; };
  size_t ws_bias = 0;  // bias-gradient partial sums, one scratch slice per (layer, direction)
  int bias_slices = 1;
  struct UL { size_t wx, wh, bx, bh; };  // element offsets in the user weight vector
  std::vector<PL> pl;
  std::vector<RL> rl;
  std::vector<WL> wl;
  std::vector<UL> ul;
  size_t ws_err = 0;
  size_t ws_arrive = 0;  // persistent recurrence: per-timestep arrival counters
  size_t ws_hx = 0;      // persistent recurrence, cluster exchange: tagged h words [2][B*H/2]
  size_t ws_dtop = 0;    // bidirectional: the two halves of dy, [2][T][B][H] storage type
  size_t ws_dxacc = 0;   // bidirectional bf16: dx of both directions summed in f32, [T][B][I]
  int ctr_count = 0;
  // streams and events (created on first use)
  std::vector<cudaStream_t> streams;
  std::vector<cudaEvent_t> ev;  // [layer][chunk]
  cudaEvent_t ev_fork = nullptr;
  std::vector<cudaEvent_t> ev_join;
  Profiler* prof = nullptr;
  // launch sequences captured as CUDA graphs, keyed by call kind and pointers
  struct GraphEntry {
    std::vector<uintptr_t> key;
    cudaGraphExec_t exec = nullptr;
    std::vector<Profiler::Rec> prof;
    unsigned long long kernels = 0;
  };
  std::vector<GraphEntry> graphs;
  std::vector<std::vector<uintptr_t>> seen, no_graph;
  cudaStream_t cap = nullptr;

  int In(int l) const { return l == 0 ? d.input : D * d.hidden; }
  int V() const { return d.layers * D; }
};

namespace {

size_t take(size_t& cur, size_t bytes) {
  const size_t at = (cur + 255) & ~size_t(255);
  cur = at + bytes;
  return at;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int plan_and_layout(rnn_s* h) {
  const rnn_desc_t& d = h->d;
  const int L = d.layers, T = d.T, B = d.B, H = d.hidden;
  h->G = d.cell == RNN_LSTM ? 4 : d.cell == RNN_GRU ? 3 : 1;
  h->GH = h->G * H;
  h->D = (d.flags & RNN_FLAG_BIDIRECTIONAL) ? 2 : 1;
  h->elem = d.mode == RNN_MODE_BF16 ? 2 : 4;
  const int GH = h->GH;
  if (d.mode == RNN_MODE_BF16) {
    if (H % 64 || d.input % 8) return RNN_ERR_UNSUPPORTED;
    const bool simple = d.cell == RNN_TANH || d.cell == RNN_RELU;
    h->u = (simple && H % 128 == 0) ? 128 : 64;
    // a forward step has ceil(B/128) x H/u tiles: narrow the packing unit
    // (down to 16 units, 32 for tanh) until a step covers at least 64 CTAs
    const int mtl = (B + 127) / 128, umin = simple ? 32 : 16;
    while (h->u > umin && mtl * (H / h->u) < 64) h->u /= 2;
  } else {
    if (H % 32 || d.input % 4) return RNN_ERR_UNSUPPORTED;
    h->u = 32;
  }
  h->limit_ns = d.timeout_ns > 0 ? (uint64_t)d.timeout_ns : 2000000000ull;

  // persistent recurrence for small batches (weights on-chip, one launch per
  // layer): whether it fits is found here, whether it is taken after the
  // stacked plans below (it runs layer after layer and replaces the
  // wavefront; for several layers the stacked recurrences, which overlap the
  // layers, measured faster).
  // (bidirectional stacks: one launch per direction, the reverse one walking time backwards)
  bool pfits = false;
  int p_ctas = 0, p_cl = 0;
  if (d.mode == RNN_MODE_BF16 && !(d.flags & (RNN_FLAG_FORCE_STREAMING | RNN_FLAG_FORCE_STACK))) {
    p_cl = 4;  // without a device: the size that co-resides on GB300 for 128 CTAs
    pfits = h->have_device ? persist_check(d.cell, H, B, h->num_sms, &p_ctas, &p_cl) == RNN_OK
                           : (B <= 8 && H % 128 == 0 && H <= (d.cell == RNN_TANH || d.cell == RNN_RELU ? 2048 : 1024));
  }
  if ((d.flags & RNN_FLAG_FORCE_PERSISTENT) && !pfits) return RNN_ERR_UNSUPPORTED;
  const bool persist_first = pfits && ((d.flags & RNN_FLAG_FORCE_PERSISTENT) || L == 1 || h->D == 2);
  if (persist_first) {
    h->persist = h->persist_plan = 1;
    h->persist_ctas = p_ctas;
    h->persist_cl = (d.flags & RNN_FLAG_NO_PERSIST_CLUSTER) ? 0 : p_cl;
  }
  // fp8 stash of W_h for the persistent inference recurrence (wider layers on chip)
  if (d.flags & RNN_FLAG_FP8_STASH) {
    if (d.mode != RNN_MODE_BF16 || (d.flags & RNN_FLAG_FORCE_STREAMING)) return RNN_ERR_UNSUPPORTED;
    int ctas = 0, cl = 0;
    const bool simple = d.cell == RNN_TANH || d.cell == RNN_RELU;
    bool fits;
    if (h->have_device) {
      fits = persist_check(d.cell, H, B, h->num_sms, &ctas, &cl, true) == RNN_OK;
    } else {  // host-side planning: the sizes the device check accepts on GB300
      fits = B <= 8 && H % 128 == 0 && H <= (simple ? 4096 : 2048);
      for (int c = 2; c <= 8 && fits; c *= 2)
        if ((H / 2) * B / c <= 1024) { cl = c; break; }
    }
    if (!fits) return RNN_ERR_UNSUPPORTED;
    h->persist8 = 1;
    h->persist8_cl = (d.flags & RNN_FLAG_NO_PERSIST_CLUSTER) ? 0 : cl;
  }
  // wavefront chunking
  // (a bidirectional layer needs all of the layer below: no wavefront)
  h->wavefront = (L > 1) && !(d.flags & RNN_FLAG_NO_WAVEFRONT) && !h->persist && h->D == 1;
  if (!h->wavefront) h->chunk = T;
  else if (d.chunk > 0) h->chunk = std::min(d.chunk, T);
  else h->chunk = std::max(1, (T + 7) / 8);
  h->nch = (T + h->chunk - 1) / h->chunk;

  // Transposed recurrent steps: with at most 256 batch entries, W_h h^T puts
  // the batch on the tile columns and keeps the epilogue's accesses
  // contiguous.  Where it wins was measured over batch (1..512) and width
  // (256..8192) on one-layer training steps: LSTM from H = 2048 at every batch
  // size, from H = 1024 at B >= 64 and from H = 256 for 64 <= B <= 128; tanh
  // RNN from H = 2048.
  if (d.mode == RNN_MODE_BF16 && !h->persist && d.cell != RNN_GRU && B <= 256 &&
      H % 32 == 0 && !(d.flags & RNN_FLAG_NO_TRANSPOSED)) {
    const bool lstm_wins = d.cell == RNN_LSTM && (H >= 2048 || (H >= 1024 && B >= 64) ||
                                                   (H >= 256 && B >= 64 && B <= 128));
    const bool tanh_wins = (d.cell == RNN_TANH || d.cell == RNN_RELU) && H >= 2048;
    if (lstm_wins || tanh_wins || (d.flags & RNN_FLAG_FORCE_TRANSPOSED)) h->tstep = 1;
  }
  if ((d.flags & RNN_FLAG_FORCE_TRANSPOSED) && !h->tstep) return RNN_ERR_UNSUPPORTED;
  if (h->tstep) {
    h->u = 1;
    h->slim_step = (d.cell == RNN_LSTM && B > 128 && (d.flags & RNN_FLAG_SLIM_STEP)) ? 1 : 0;
    // several steps per launch: one tile of 256 gate rows x the batch per SM pair and step
    const int sbn = B > 128 ? 256 : B > 64 ? 128 : 64;
    h->step_chunks = (d.cell == RNN_LSTM && !h->slim_step && h->D == 1 && B % 32 == 0 &&
                      ((GH + 255) / 256) * ((B + sbn - 1) / sbn) <= h->num_sms / 2 &&
                      (d.flags & RNN_FLAG_STEP_CHUNKS)) ? 1 : 0;
    // backward: 128-unit x bn-batch tiles, K split in clusters of a power of
    // two that the K blocks fill exactly, until the step covers the SMs
    h->bwd_bn = B > 128 ? 256 : B > 64 ? 128 : 64;
    const int tiles = (H + 127) / 128;
    const int kb = (GH + 63) / 64;
    int s = 1;
    while (s * 2 <= 8 && tiles * s * 2 <= h->num_sms && h->bwd_bn % (16 * s * 2) == 0 && kb / (s * 2) >= 4 &&
           (s * 2 - 1) * ((kb + s * 2 - 1) / (s * 2)) < kb)
      s *= 2;
    h->bwd_splits = s;
    h->ctr_count = tiles;
    h->bwd_fuse = (d.cell == RNN_LSTM && h->bwd_bn == 256 && s == 4 && !(d.flags & RNN_FLAG_NO_FUSED_POINT)) ? 1 : 0;
  } else if (d.mode == RNN_MODE_BF16) {
    // backward step tiles: 128-row batch tiles x bn hidden units, split over K
    // until the step covers the SMs (at most 8 ways, at least 4 K blocks each)
    h->bwd_bn = (H % 256 == 0) ? 256 : 128;
    // narrower tiles when even 8-way splits of 256-wide tiles leave most SMs idle
    if (h->bwd_bn == 256 && ((B + 127) / 128) * (H / 256) * 8 < h->num_sms / 2) h->bwd_bn = 128;
    const int tiles = ((B + 127) / 128) * ((H + h->bwd_bn - 1) / h->bwd_bn);
    const int kb = (GH + 63) / 64;
    int want = std::max(1, h->num_sms / std::max(1, tiles));
    want = std::min(want, 8);
    want = std::min(want, std::max(1, kb / 4));
    // a power of two that the K blocks fill exactly, so that every split has
    // work and the cluster reduction cuts the tile into 16-column slices
    int s = 1;
    while (s * 2 <= want && (s * 2 - 1) * ((kb + s * 2 - 1) / (s * 2)) < kb) s *= 2;
    h->bwd_splits = s;
    h->ctr_count = tiles;
  } else {
    h->bwd_bn = 32;
    h->bwd_splits = 1;
    h->ctr_count = 1;
  }

  // persistent stacked forward for moderate batches: the layers in groups of
  // up to kStackMaxLayers that fit on the device together
  if (d.mode == RNN_MODE_BF16 && h->D == 1 && !h->persist && B <= 64 &&
      !(d.flags & (RNN_FLAG_NO_STACK | RNN_FLAG_FORCE_STREAMING))) {
    const int sms = h->have_device ? h->num_sms : 0;
    int wide = 0;  // the last group checked needs chunks wider than TMEM holds
    auto fits = [&](int l0, int nl) {
      int ctas = 0;
      return stack_check(d.cell, H, B, nl, l0 == 0 ? 1 : 0, h->u, sms, &ctas, &wide) == RNN_OK;
    };
    std::vector<std::pair<int, int>> groups;
    bool ok = true, overlap = false;
    for (int l0 = 0; l0 < L && ok;) {
      int nl = 0;
      while (l0 + nl < L && nl < kStackMaxLayers && fits(l0, nl + 1)) ++nl;
      if (nl == 0) ok = false;
      else groups.emplace_back(l0, nl);
      if (nl > 1) {
        fits(l0, nl);
        overlap = overlap || !wide;
      }
      l0 += nl;
    }
    // up to 8 sequences the single-layer persistent recurrence, where it
    // fits, keeps the forward unless a stacked group overlaps layers on
    // chunks that fit TMEM (measured at B <= 8, LSTM and GRU H=1024, 4
    // layers: one-layer groups and two-layer groups on widened chunks both
    // lost to the persistent forward; H <= 512 four-layer groups won 5-6x).
    // Where it does not fit (LSTM and GRU H=2048) the stacked forward beat
    // the step launches (one layer, T=16: 0.58 against 0.69 ms).
    if (B <= 8 && !overlap && pfits && !(d.flags & RNN_FLAG_FORCE_STACK)) ok = false;
    if (ok) {
      h->stack = h->stack_plan = 1;
      h->stack_groups = groups;
    }
  }
  if ((d.flags & RNN_FLAG_FORCE_STACK) && !h->stack) return RNN_ERR_UNSUPPORTED;
  if (!h->persist && !h->stack && pfits) {
    // no stacked plan fits: the single-layer persistent recurrence after all
    // (layer after layer, no wavefront)
    h->persist = h->persist_plan = 1;
    h->persist_ctas = p_ctas;
    h->persist_cl = (d.flags & RNN_FLAG_NO_PERSIST_CLUSTER) ? 0 : p_cl;
    h->wavefront = 0;
    h->chunk = T;
    h->nch = 1;
  }
  // persistent stacked backward, same batch range: groups of up to
  // kStackMaxLayers layers from the top of the stack down
  if (d.mode == RNN_MODE_BF16 && h->D == 1 && B <= 64 &&
      !(d.flags & (RNN_FLAG_NO_STACK | RNN_FLAG_NO_STACK_BWD | RNN_FLAG_FORCE_STREAMING | RNN_FLAG_FORCE_PERSISTENT))) {
    const int sms = h->have_device ? h->num_sms : 0;
    std::vector<std::pair<int, int>> groups;
    std::vector<int> budgets;
    bool ok = true;
    for (int top = L - 1; top >= 0 && ok;) {
      int nl = 0, budget = 0;
      while (top - nl >= 0 && nl < kStackMaxLayers) {
        int ctas = 0, b = 0;
        if (stack_bwd_check(d.cell, H, B, nl + 1, top == L - 1 ? 1 : 0, h->u, sms, &ctas, &b) != RNN_OK) break;
        ++nl;
        budget = b;
      }
      if (nl == 0) ok = false;
      else {
        groups.emplace_back(top - nl + 1, nl);
        budgets.push_back(budget);
      }
      top -= nl;
    }
    // Recurrent-only tops: each group's top layer runs only its recurrent
    // product in the kernel, the gradient from the layer above (computed by
    // the group before) entering as one GEMM over all steps; the layers below
    // it in the group take the share from above in the kernel as usual.  It
    // needs fewer CTAs where the share from above does not fit beside the
    // recurrent one (K = 2 G H); taken when the full groups do not fit or
    // it makes fewer groups.
    std::vector<std::pair<int, int>> rgroups;
    std::vector<int> rbudgets;
    bool rok = true;
    for (int top = L - 1; top >= 0 && rok;) {
      int nl = 0, budget = 0;
      while (top - nl >= 0 && nl < kStackMaxLayers) {
        int ctas = 0, b = 0;
        if (stack_bwd_check(d.cell, H, B, nl + 1, 1, h->u, sms, &ctas, &b) != RNN_OK) break;
        ++nl;
        budget = b;
      }
      if (nl == 0) rok = false;
      else {
        rgroups.emplace_back(top - nl + 1, nl);
        rbudgets.push_back(budget);
      }
      top -= nl;
    }
    if (rok && (!ok || rgroups.size() < groups.size())) {
      groups = rgroups;
      budgets = rbudgets;
      ok = true;
      h->stackb_rec = 1;
    }
    if (ok) {
      h->stackb = h->stackb_plan = 1;
      h->stackb_groups = groups;
      h->stackb_budget = budgets;
    }
  }

  const size_t e = h->elem;
  const size_t BH = (size_t)B * H, BGH = (size_t)B * GH;
  // per (layer, direction) v = l * D + d; In of layer l = v / D
  const int V = h->V(), Dn = h->D;
  // user weights
  h->ul.resize(V);
  size_t off = 0;
  for (int l = 0; l < V; ++l) {
    h->ul[l].wx = off; off += (size_t)GH * h->In(l / Dn);
    h->ul[l].wh = off; off += (size_t)GH * H;
    h->ul[l].bx = off; off += GH;
    h->ul[l].bh = off; off += GH;
  }
  h->user_w_bytes = off * e;
  // packed weights
  h->pl.resize(V);
  size_t cur = 0;
  for (int l = 0; l < V; ++l) {
    h->pl[l].wx = take(cur, (size_t)GH * h->In(l / Dn) * e);
    h->pl[l].wh = take(cur, (size_t)GH * H * e);
    h->pl[l].bias = take(cur, (size_t)GH * 4);
    h->pl[l].bias_hn = take(cur, (size_t)H * 4);
    h->pl[l].wh8 = (d.flags & RNN_FLAG_FP8_STASH) ? take(cur, (size_t)GH * H) : 0;
    h->pl[l].wsc = (d.flags & RNN_FLAG_FP8_STASH) ? take(cur, (size_t)GH * 4) : 0;
  }
  h->packed_bytes = (cur + 255) & ~size_t(255);
  // reserve
  h->rl.resize(V);
  cur = 0;
  for (int l = 0; l < V; ++l) {
    h->rl[l].gates = take(cur, (size_t)T * BGH * 4);
    h->rl[l].c = d.cell == RNN_LSTM ? take(cur, (size_t)T * BH * 4) : 0;
    h->rl[l].hn = d.cell == RNN_GRU ? take(cur, (size_t)T * BH * 4) : 0;
    h->rl[l].hseq = take(cur, (size_t)(T + 1) * BH * e);
    h->rl[l].dgx = take(cur, (size_t)T * BGH * e);
    h->rl[l].dgh = d.cell == RNN_GRU ? take(cur, (size_t)T * BGH * e) : h->rl[l].dgx;
  }
  h->reserve_bytes = (cur + 255) & ~size_t(255);
  // workspace
  h->wl.resize(V);
  cur = 0;
  h->ws_err = take(cur, 256);
  h->ws_arrive = take(cur, (size_t)std::max(kStackMaxLayers, L) * T * 4);  // per-timestep counters (stack: a row per layer)
  h->ws_hx = (h->persist_plan || h->persist8) ? take(cur, (size_t)8 * B * H) : 0;
  h->bias_slices = std::max(1, std::min(64, (T * B + 255) / 256));
  h->ws_bias = take(cur, (size_t)V * h->bias_slices * GH * 4);  // one scratch slice per (layer, direction)
  h->ws_dtop = Dn == 2 ? take(cur, (size_t)2 * T * BH * e) : 0;
  h->ws_dxacc = (Dn == 2 && d.mode == RNN_MODE_BF16) ? take(cur, (size_t)T * B * d.input * 4) : 0;
  for (int l = 0; l < V; ++l) {
    h->wl[l].P = take(cur, (size_t)T * BGH * 4);
    h->wl[l].hseq = take(cur, (size_t)(T + 1) * BH * e);
    h->wl[l].c2 = take(cur, 2 * BH * 4);
    h->wl[l].dyab = take(cur, (size_t)T * BH * 4);
    h->wl[l].carry = take(cur, BH * 4);
    // split-K partials; the transposed product pads each split's batch rows to whole tiles
    const size_t bp = h->tstep ? (size_t)((B + h->bwd_bn - 1) / h->bwd_bn * h->bwd_bn) : (size_t)B;
    h->wl[l].part = take(cur, (size_t)h->bwd_splits * bp * H * 4);
    h->wl[l].dh = h->tstep ? take(cur, BH * 4) : 0;
    h->wl[l].ctr = take(cur, (size_t)h->ctr_count * 4);
  }
  h->ws_bytes = (cur + 255) & ~size_t(255);
  return RNN_OK;
}

int ensure_runtime(rnn_s* h) {
  if (!h->have_device) return RNN_ERR_CUDA;
  if (!h->streams.empty() || h->d.layers == 0) return RNN_OK;
  const int L = h->d.layers;
  const int NS = std::max(L, h->D);  // one stream per layer (wavefront) or per direction
  h->streams.resize(NS);
  for (int l = 0; l < NS; ++l)
    if (cudaStreamCreateWithFlags(&h->streams[l], cudaStreamNonBlocking) != cudaSuccess) return RNN_ERR_CUDA;
  h->ev.resize((size_t)L * h->nch);
  for (auto& e : h->ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return RNN_ERR_CUDA;
  if (cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess) return RNN_ERR_CUDA;
  h->ev_join.resize(NS);
  for (auto& e : h->ev_join)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return RNN_ERR_CUDA;
  return RNN_OK;
}

// fork the layer streams off the caller's stream / join them back
int fork_streams(rnn_s* h, cudaStream_t s) {
  if (cudaEventRecord(h->ev_fork, s) != cudaSuccess) return RNN_ERR_CUDA;
  for (auto st : h->streams)
    if (cudaStreamWaitEvent(st, h->ev_fork, 0) != cudaSuccess) return RNN_ERR_CUDA;
  return RNN_OK;
}
int join_streams(rnn_s* h, cudaStream_t s) {
  for (size_t l = 0; l < h->streams.size(); ++l) {
    if (cudaEventRecord(h->ev_join[l], h->streams[l]) != cudaSuccess) return RNN_ERR_CUDA;
    if (cudaStreamWaitEvent(s, h->ev_join[l], 0) != cudaSuccess) return RNN_ERR_CUDA;
  }
  return RNN_OK;
}

Launch mk(rnn_s* h, cudaStream_t s, void* ws, const char* name) {
  Launch L;
  L.stream = s;
  L.err = ws ? reinterpret_cast<int*>(static_cast<char*>(ws) + h->ws_err) : nullptr;
  L.limit_ns = h->limit_ns;
  L.num_sms = h->num_sms;
  L.prof = (h->d.flags & RNN_FLAG_PROFILE) ? h->prof : nullptr;
  L.name = name;
  L.pair = (h->d.flags & RNN_FLAG_NO_PAIR) ? 0 : 1;
  // per-kernel event timing needs each kernel to start after the previous one.
  // A programmatic dependent launch lets the next kernel on a stream take
  // SMs while the previous one drains; in the layer wavefront of the step
  // launches another layer's kernel can use them instead, which measured
  // faster (4-layer LSTM H=4096 B=256 training step: 33.6 ms without, 34.1
  // ms with, three alternating runs each), so only a single stream of
  // launches (one layer, or the wavefront off) is launched dependently.
  L.pdl = ((h->d.flags & (RNN_FLAG_NO_PDL | RNN_FLAG_PROFILE)) || (h->wavefront && !h->stack)) ? 0 : 1;
  return L;
}

// Runs `issue` (which enqueues a whole call on the stream it is given) through
// a cached CUDA graph: the first call with a given key runs directly, the
// second is captured (on an internal stream, with the layer streams forked
// from it) and every later one replays the graph on the caller's stream, so a
// call costs one graph launch instead of hundreds of kernel launches.  A
// capture that fails leaves the key on the direct path.
template <class F>
int run_graphed(rnn_s* h, cudaStream_t user, const std::vector<uintptr_t>& key, F&& issue) {
  if (h->d.flags & RNN_FLAG_NO_GRAPH) return issue(user);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(user, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return issue(user);
  for (auto& g : h->graphs) {
    if (g.key != key) continue;
    if (cudaGraphLaunch(g.exec, user) != cudaSuccess) return RNN_ERR_CUDA;
    g_launches += g.kernels;
    if (h->prof && (h->d.flags & RNN_FLAG_PROFILE)) {
      std::lock_guard<std::mutex> lk(h->prof->mu);
      for (auto& r : g.prof) {
        h->prof->pending.push_back(r);
      }
    }
    return RNN_OK;
  }
  auto in = [&](const std::vector<std::vector<uintptr_t>>& v) { return std::find(v.begin(), v.end(), key) != v.end(); };
  if (in(h->no_graph)) return issue(user);
  if (!in(h->seen)) {
    if (h->seen.size() >= 64) h->seen.erase(h->seen.begin());
    h->seen.push_back(key);
    return issue(user);
  }
  if (!h->cap && cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking) != cudaSuccess) return issue(user);
  const unsigned long long before = g_launches.load();
  if (cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    h->no_graph.push_back(key);
    return issue(user);
  }
  if (h->prof) {
    std::lock_guard<std::mutex> lk(h->prof->mu);
    h->prof->capturing = true;
    h->prof->captured.clear();
  }
  const int rc = issue(h->cap);
  cudaGraph_t gr = nullptr;
  const cudaError_t e = cudaStreamEndCapture(h->cap, &gr);
  std::vector<Profiler::Rec> recs;
  if (h->prof) {
    std::lock_guard<std::mutex> lk(h->prof->mu);
    h->prof->capturing = false;
    recs.swap(h->prof->captured);
  }
  const unsigned long long kernels = g_launches.load() - before;
  g_launches -= kernels;  // captured, not run
  cudaGraphExec_t ex = nullptr;
  const bool ok = rc == RNN_OK && e == cudaSuccess && gr && cudaGraphInstantiate(&ex, gr, 0) == cudaSuccess;
  if (gr) cudaGraphDestroy(gr);
  if (!ok) {
    cudaGetLastError();
    for (auto& r : recs) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    h->no_graph.push_back(key);
    return issue(user);
  }
  if (h->graphs.size() >= 8) {  // evict the oldest (let it finish first)
    cudaDeviceSynchronize();
    cudaGraphExecDestroy(h->graphs.front().exec);
    for (auto& r : h->graphs.front().prof) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    h->graphs.erase(h->graphs.begin());
  }
  rnn_s::GraphEntry ge;
  ge.key = key;
  ge.exec = ex;
  ge.prof = std::move(recs);
  ge.kernels = kernels;
  h->graphs.push_back(std::move(ge));
  auto& g = h->graphs.back();
  if (cudaGraphLaunch(g.exec, user) != cudaSuccess) return RNN_ERR_CUDA;
  g_launches += g.kernels;
  if (h->prof && (h->d.flags & RNN_FLAG_PROFILE)) {
    std::lock_guard<std::mutex> lk(h->prof->mu);
    for (auto& r : g.prof) h->prof->pending.push_back(r);
  }
  return RNN_OK;
}

#define RNN_TRY(x)              \
  do {                          \
    int rc__ = (x);             \
    if (rc__ != RNN_OK) return rc__; \
  } while (0)

int cu(cudaError_t e) { return e == cudaSuccess ? RNN_OK : RNN_ERR_CUDA; }

// Copies and zero fills inside a call run as kernels on the call's stream
// (dev_copy, dev_zero): never as copy-engine operations, which would wait
// behind a large transfer the caller keeps on a copy engine.
int zero_async(rnn_s* h, void* p, size_t n, cudaStream_t s) { return dev_zero(mk(h, s, nullptr, "fill"), p, n); }
int copy_async(rnn_s* h, void* d, const void* src, size_t n, cudaStream_t s) {
  return dev_copy(mk(h, s, nullptr, "copy"), d, src, n);
}
int copy2d_async(rnn_s* h, void* d, size_t dp, const void* src, size_t sp, size_t w, size_t rows, cudaStream_t s) {
  return dev_copy2d(mk(h, s, nullptr, "copy"), d, dp, src, sp, w, rows);
}

// ---------------------------------------------------------------- bidirectional stacks
// Every layer has a forward (d = 0) and a reverse (d = 1) direction with their
// own weights, v = 2 l + d.  Both keep their h sequence in time order: the
// forward one at slots 1..T (slot 0 = its h0), the reverse one at slots
// 0..T-1 (slot T = its h0), so the next layer's input, dW_x and dW_h read
// plain strided operands.  A layer's input of width 2H enters its products as
// two halves of K (the second product accumulating).  Layers run one after
// another (layer l + 1 needs all of layer l's reverse direction); the two
// directions of a layer run side by side on two streams, forked from and
// joined back into the caller's stream around each layer.

// hand-off cluster size of the persistent recurrence (0: counters), bf16 or fp8-stash plan
int pa_cluster(const rnn_s* h, bool p8) { return p8 ? h->persist8_cl : h->persist_cl; }

// Backward data pass with the persistent stacked recurrence: one launch per
// layer group from the top of the stack down (each computes its layers' gate
// gradients, dh0 and dc0), then the gradient of the stack's input dGx^0 W_x^0
// as one GEMM over all timesteps.
int bwd_stack(rnn_s* h, const void* dy, const void* dhT, const float* dcT, const char* PW, const float* c0, void* dx,
              void* dh0, float* dc0, char* R, char* W, void* ws, cudaStream_t stream) {
  const rnn_desc_t& d = h->d;
  const int L = d.layers, T = d.T, B = d.B, H = d.hidden, GH = h->GH;
  const size_t e = h->elem, BH = (size_t)B * H, BGH = (size_t)B * GH;
  const bool lstm = d.cell == RNN_LSTM, gru = d.cell == RNN_GRU;
  // one counter row per layer, zeroed once for all groups
  unsigned int* cnt = reinterpret_cast<unsigned int*>(W + h->ws_arrive);
  RNN_TRY(zero_async(h, cnt, (size_t)L * T * 4, stream));
  for (size_t gi = 0; gi < h->stackb_groups.size(); ++gi) {
    const int l0 = h->stackb_groups[gi].first, nl = h->stackb_groups[gi].second;
    // recurrent-only groups: the gradient reaching this layer's outputs from
    // the layer above, dGx^{l+1} W_x^{l+1}, as one product over all steps
    const int lt = l0 + nl - 1;  // the group's top layer
    float* dyab = nullptr;
    if (h->stackb_rec && lt < L - 1) {
      dyab = reinterpret_cast<float*>(W + h->wl[lt].dyab);
      Operand A{R + h->rl[lt + 1].dgx, GH, 0, T * B, GH};
      Operand Bx{PW + h->pl[lt + 1].wx, H, 1, H, GH, 1};
      Remap none{0, 1, 1, 1};
      Launch Lg = mk(h, stream, ws, "dx_gemm");
      RNN_TRY(gemm_f32(Lg, d.mode, A, Bx, T * B, H, GH, dyab, H, nullptr, 0, none, 0));
    }
    StackBwdArgs sa{};
    sa.budget = h->stackb_budget[gi];
    sa.T = T;
    sa.B = B;
    sa.H = H;
    sa.u_pack = h->u;
    sa.nl = nl;
    for (int i = 0; i < nl; ++i) {
      const int l = l0 + i;
      const bool top = l == L - 1 || (h->stackb_rec && l == lt);  // no layer above inside the kernel
      StackBwdLayer& ly = sa.lay[i];
      ly.Wh = reinterpret_cast<const __nv_bfloat16*>(PW + h->pl[l].wh);
      ly.Wx_above = top ? nullptr : reinterpret_cast<const __nv_bfloat16*>(PW + h->pl[l + 1].wx);
      ly.dgx = reinterpret_cast<__nv_bfloat16*>(R + h->rl[l].dgx);
      ly.dgh = reinterpret_cast<__nv_bfloat16*>(R + h->rl[l].dgh);
      ly.dgx_above = top ? nullptr : reinterpret_cast<const __nv_bfloat16*>(R + h->rl[l + 1].dgx);
      ly.gates = reinterpret_cast<const float*>(R + h->rl[l].gates);
      ly.c = lstm ? reinterpret_cast<const float*>(R + h->rl[l].c) : nullptr;
      ly.c0 = (lstm && c0) ? c0 + l * BH : nullptr;
      ly.hn = gru ? reinterpret_cast<const float*>(R + h->rl[l].hn) : nullptr;
      ly.hseq = reinterpret_cast<const __nv_bfloat16*>(R + h->rl[l].hseq);
      ly.dy = l == L - 1 ? dy : l == lt ? dyab : nullptr;
      ly.dy_f32 = l == L - 1 ? 0 : 1;
      ly.dhT = dhT ? reinterpret_cast<const __nv_bfloat16*>(static_cast<const char*>(dhT) + l * BH * e) : nullptr;
      ly.dcT = (lstm && dcT) ? dcT + l * BH : nullptr;
      ly.dh0 = dh0 ? reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(dh0) + l * BH * e) : nullptr;
      ly.dc0 = (lstm && dc0) ? dc0 + l * BH : nullptr;
      ly.wait_above = i + 1 < nl ? 1 : 0;
    }
    sa.cnt = cnt + (size_t)l0 * T;
    sa.err = reinterpret_cast<int*>(W + h->ws_err);
    sa.limit_ns = h->limit_ns;
    sa.test_skip_publish = (d.flags & RNN_FLAG_TEST_SKIP_PUBLISH) ? 1 : 0;
    Launch Lk = mk(h, stream, ws, "stack_bwd");
    RNN_TRY(stack_bwd(Lk, d.cell, sa));
  }
  if (dx) {
    Operand A{R + h->rl[0].dgx, GH, 0, T * B, GH};
    Operand Bx{PW + h->pl[0].wx, d.input, 1, d.input, GH, 1};
    Launch Lk = mk(h, stream, ws, "dx_gemm");
    RNN_TRY(gemm_store(Lk, d.mode, A, Bx, T * B, d.input, GH, dx, d.input, 0));
  }
  (void)BGH;
  return RNN_OK;
}

// Forward pass with the persistent stacked recurrence: layer 0's input
// projection for all timesteps as one GEMM, then one launch per layer group.
int fwd_stack(rnn_s* h, const void* x, const void* h0, const float* c0, const char* PW, void* y, void* hT, float* cT,
              char* R, char* W, void* ws, cudaStream_t stream) {
  const rnn_desc_t& d = h->d;
  const int L = d.layers, T = d.T, B = d.B, H = h->d.hidden, GH = h->GH;
  const size_t e = h->elem, BH = (size_t)B * H, BGH = (size_t)B * GH;
  const bool train = R != nullptr;
  const bool lstm = d.cell == RNN_LSTM, gru = d.cell == RNN_GRU;
  auto hseq_of = [&](int l) { return train ? R + h->rl[l].hseq : W + h->wl[l].hseq; };
  float* P0 = reinterpret_cast<float*>(train ? R + h->rl[0].gates : W + h->wl[0].P);
  {
    Operand A{x, d.input, 0, T * B, d.input};
    Operand Bw{PW + h->pl[0].wx, d.input, 0, GH, d.input, 1};
    Remap none{0, 1, 1, 1};
    Launch Lk = mk(h, stream, ws, "input_proj_gemm");
    RNN_TRY(gemm_f32(Lk, d.mode, A, Bw, T * B, GH, d.input, P0, GH, reinterpret_cast<const float*>(PW + h->pl[0].bias),
                     0, none, 0));
  }
  // every layer's h_{-1} and every layer's counter row (one per layer, so
  // that the groups need no zeroing between them) in one launch
  unsigned int* cnt = reinterpret_cast<unsigned int*>(W + h->ws_arrive);
  {
    std::vector<DevOp> ops;
    for (int l = 0; l < L; ++l) ops.push_back({hseq_of(l), h0 ? static_cast<const char*>(h0) + l * BH * e : nullptr, BH * e});
    ops.push_back({cnt, nullptr, (size_t)L * T * 4});
    RNN_TRY(dev_batch(mk(h, stream, nullptr, "copy"), ops.data(), (int)ops.size()));
  }
  for (const auto& grp : h->stack_groups) {
    const int l0 = grp.first, nl = grp.second;
    StackArgs sa{};
    sa.T = T;
    sa.B = B;
    sa.H = H;
    sa.u_pack = h->u;
    sa.nl = nl;
    for (int i = 0; i < nl; ++i) {
      const int l = l0 + i;
      char* hs = hseq_of(l);
      StackLayer& ly = sa.lay[i];
      ly.Wx = l > 0 ? reinterpret_cast<const __nv_bfloat16*>(PW + h->pl[l].wx) : nullptr;
      ly.Wh = reinterpret_cast<const __nv_bfloat16*>(PW + h->pl[l].wh);
      ly.P = l == 0 ? P0 : nullptr;
      ly.bias = reinterpret_cast<const float*>(PW + h->pl[l].bias);
      ly.bias_hn = reinterpret_cast<const float*>(PW + h->pl[l].bias_hn);
      ly.c0 = (lstm && c0) ? c0 + l * BH : nullptr;
      ly.gates_out = train ? reinterpret_cast<float*>(R + h->rl[l].gates) : nullptr;
      ly.c_out = (train && lstm) ? reinterpret_cast<float*>(R + h->rl[l].c) : nullptr;
      ly.hn_out = (train && gru) ? reinterpret_cast<float*>(R + h->rl[l].hn) : nullptr;
      ly.hseq = reinterpret_cast<__nv_bfloat16*>(hs);
      ly.in = l > 0 ? reinterpret_cast<const __nv_bfloat16*>(hseq_of(l - 1)) : nullptr;
      ly.y = l == L - 1 ? static_cast<__nv_bfloat16*>(y) : nullptr;
      ly.hT = hT ? reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(hT) + (size_t)l * BH * e) : nullptr;
      ly.cT = (cT && lstm) ? cT + (size_t)l * BH : nullptr;
      ly.In = l > 0 ? H : d.input;
      ly.wait_in = i > 0 ? 1 : 0;
    }
    sa.cnt = cnt + (size_t)l0 * T;
    sa.err = reinterpret_cast<int*>(W + h->ws_err);
    sa.limit_ns = h->limit_ns;
    sa.test_skip_publish = (d.flags & RNN_FLAG_TEST_SKIP_PUBLISH) ? 1 : 0;
    Launch Lk = mk(h, stream, ws, "stack_fwd");
    RNN_TRY(stack_fwd(Lk, d.cell, sa));
  }
  return RNN_OK;
}

// slot of h at time t in direction d (t = -1 forward, t = T reverse: the initial state)
size_t hslot(int d, int t) { return (size_t)(t + 1 - d); }

int fwd_bidir(rnn_s* h, const void* x, const void* h0, const float* c0, const char* PW, void* y, void* hT,
              float* cT, char* R, char* W, void* ws, cudaStream_t s) {
  const rnn_desc_t& d = h->d;
  const int L = d.layers, T = d.T, B = d.B, H = d.hidden, GH = h->GH, mode = d.mode;
  const size_t e = h->elem, BH = (size_t)B * H, BGH = (size_t)B * GH;
  const bool train = R != nullptr;
  const bool lstm = d.cell == RNN_LSTM, gru = d.cell == RNN_GRU;
  const Remap none{0, 1, 1, 1};
  auto hseq_of = [&](int v) -> char* { return train ? R + h->rl[v].hseq : W + h->wl[v].hseq; };
  cudaStream_t caller = s;
  // directions side by side (not the persistent recurrence: two grids that
  // each need most of the SMs at once must not be launched together)
  const bool p8 = !train && h->persist8 && h->varlen == 0;  // fp8 stash (inference)
  const bool pers = p8 || h->persist;
  const bool side = !(d.flags & RNN_FLAG_NO_WAVEFRONT) && !pers;
  // variable lengths: running sequences at time t are rows 0 .. Bt[t]-1 in
  // both directions; idle positions of y and of the h sequences read 0
  const bool vl = h->varlen != 0;
  auto Bt = [&](int t) { return vl ? h->Bt[t] : (t < T ? B : 0); };
  if (vl) {
    RNN_TRY(zero_async(h, y, (size_t)T * BH * 2 * e, caller));
    for (int v = 0; v < 2 * L; ++v) RNN_TRY(zero_async(h, hseq_of(v), (size_t)(T + 1) * BH * e, caller));
  }
  for (int l = 0; l < L; ++l) {
    if (side) RNN_TRY(fork_streams(h, caller));
    for (int dd = 0; dd < 2; ++dd) {
      const int v = 2 * l + dd;
      s = side ? h->streams[dd] : caller;
      char* hseq = hseq_of(v);
      float* P = reinterpret_cast<float*>(train ? R + h->rl[v].gates : W + h->wl[v].P);
      char* hinit = hseq + hslot(dd, dd == 0 ? -1 : T) * BH * e;
      if (h0)
        RNN_TRY(copy_async(h, hinit, static_cast<const char*>(h0) + v * BH * e, BH * e, s));
      else
        RNN_TRY(zero_async(h, hinit, BH * e, s));
      // input projection over all T (layer >= 1: one product per half of the input)
      const float* bias = reinterpret_cast<const float*>(PW + h->pl[v].bias);
      if (l == 0) {
        const int In = d.input;
        Operand A{x, In, 0, T * B, In};
        Operand Bw{PW + h->pl[v].wx, In, 0, GH, In, 1};
        Launch Lk = mk(h, s, ws, "input_proj_gemm");
        RNN_TRY(gemm_f32(Lk, mode, A, Bw, T * B, GH, In, P, GH, bias, 0, none, 0));
      } else {
        for (int q = 0; q < 2; ++q) {
          Operand A{hseq_of(2 * (l - 1) + q) + hslot(q, 0) * BH * e, H, 0, T * B, H};
          Operand Bw{PW + h->pl[v].wx + (size_t)q * H * e, 2 * H, 0, GH, H, 1};
          Launch Lk = mk(h, s, ws, "input_proj_gemm");
          RNN_TRY(gemm_f32(Lk, mode, A, Bw, T * B, GH, H, P, GH, q == 0 ? bias : nullptr, q, none, 0));
        }
      }
      auto cbuf = [&](int tt) -> float* {
        return train ? reinterpret_cast<float*>(R + h->rl[v].c) + (size_t)tt * BH
                     : reinterpret_cast<float*>(W + h->wl[v].c2) + (size_t)(tt & 1) * BH;
      };
      if (pers) {
        // all T steps of this direction in one launch
        unsigned int* arrive = reinterpret_cast<unsigned int*>(W + h->ws_arrive);
        if (pa_cluster(h, p8)) RNN_TRY(zero_async(h, W + h->ws_hx, (size_t)8 * B * H, s));
        else RNN_TRY(zero_async(h, arrive, (size_t)T * 4, s));
        PersistArgs pa{};
        pa.arrive = arrive;
        pa.cluster = pa_cluster(h, p8);
        pa.cluster_sync = (d.flags & RNN_FLAG_PERSIST_CLUSTER_SYNC) ? 1 : 0;
        pa.Wh8 = p8 ? reinterpret_cast<const uint8_t*>(PW + h->pl[v].wh8) : nullptr;
        pa.wscale = p8 ? reinterpret_cast<const float*>(PW + h->pl[v].wsc) : nullptr;
        pa.hx = reinterpret_cast<uint64_t*>(W + h->ws_hx);
        pa.T = T;
        pa.B = B;
        pa.H = H;
        pa.u_pack = h->u;
        pa.Wh = reinterpret_cast<const __nv_bfloat16*>(PW + h->pl[v].wh);
        pa.P = P;
        pa.gates_out = train ? P : nullptr;
        pa.bias_hn = reinterpret_cast<const float*>(PW + h->pl[v].bias_hn);
        pa.c0 = (lstm && c0) ? c0 + v * BH : nullptr;
        pa.c_out = (train && lstm) ? reinterpret_cast<float*>(R + h->rl[v].c) : nullptr;
        pa.hn_out = (train && gru) ? reinterpret_cast<float*>(R + h->rl[v].hn) : nullptr;
        pa.hseq = reinterpret_cast<__nv_bfloat16*>(hseq);
        pa.y = nullptr;
        pa.hT = hT ? reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(hT) + (size_t)v * BH * e) : nullptr;
        pa.cT = (cT && lstm) ? cT + (size_t)v * BH : nullptr;
        pa.err = reinterpret_cast<int*>(W + h->ws_err);
        pa.limit_ns = h->limit_ns;
        pa.test_skip_publish = (d.flags & RNN_FLAG_TEST_SKIP_PUBLISH) ? 1 : 0;
        pa.reverse = dd;
        Launch Lk = mk(h, s, ws, "persist_fwd");
        RNN_TRY(persist_fwd(Lk, d.cell, pa));
      }
      // the recurrence: step k at time t, after the step at time tp
      for (int k = 0; k < T && !pers; ++k) {
        const int t = dd == 0 ? k : T - 1 - k, tp = dd == 0 ? t - 1 : t + 1;
        const int Bs = Bt(t);
        if (Bs == 0) continue;
        if (dd == 1 && vl && t < T - 1) {
          // rows Bt[t+1] .. Bs-1 start their reverse sweep here: h_prev and c_prev from h0, c0
          const int r0 = Bt(t + 1), nr = Bs - r0;
          if (nr > 0) {
            char* hp = hseq + hslot(dd, tp) * BH * e + (size_t)r0 * H * e;
            if (h0)
              RNN_TRY(copy_async(h, hp, static_cast<const char*>(h0) + (v * BH + (size_t)r0 * H) * e, (size_t)nr * H * e, s));
            else
              RNN_TRY(zero_async(h, hp, (size_t)nr * H * e, s));
            if (lstm) {
              float* cp = cbuf(tp) + (size_t)r0 * H;
              if (c0)
                RNN_TRY(copy_async(h, cp, c0 + v * BH + (size_t)r0 * H, (size_t)nr * H * 4, s));
              else
                RNN_TRY(zero_async(h, cp, (size_t)nr * H * 4, s));
            }
          }
        }
        FwdStepArgs a;
        a.B = Bs;
        a.H = H;
        a.u = h->u;
        a.P = P + (size_t)t * BGH;
        a.write_gates = train ? 1 : 0;
        a.bias_hn = reinterpret_cast<const float*>(PW + h->pl[v].bias_hn);
        a.c_prev = lstm ? (t == (dd == 0 ? 0 : T - 1) ? (c0 ? c0 + v * BH : nullptr) : cbuf(tp)) : nullptr;
        a.c_out = lstm ? cbuf(t) : nullptr;
        a.h_prev = hseq + hslot(dd, tp) * BH * e;
        a.h_out = hseq + hslot(dd, t) * BH * e;
        a.y = nullptr;
        // final states: after t = T-1 forward (or each sequence's own last
        // time, copied below), after t = 0 in reverse (every sequence runs it)
        const bool fin = dd == 0 ? (!vl && t == T - 1) : t == 0;
        a.hT = (fin && hT) ? static_cast<char*>(hT) + (size_t)v * BH * e : nullptr;
        a.cT = (fin && cT && lstm) ? cT + (size_t)v * BH : nullptr;
        a.hn_out = (train && gru) ? reinterpret_cast<float*>(R + h->rl[v].hn) + (size_t)t * BH : nullptr;
        a.slim = h->slim_step;
        Operand A{a.h_prev, H, 0, Bs, H};
        Operand Bw{PW + h->pl[v].wh, H, 0, GH, H, 1};
        Launch Lk = mk(h, s, ws, "fwd_step");
        if (h->tstep) RNN_TRY(fwd_step_t(Lk, d.cell, Bw, A, a));
        else RNN_TRY(fwd_step(Lk, mode, d.cell, A, Bw, a));
        if (dd == 0 && vl) {
          // sequences ending at time t (rows Bt[t+1] .. Bs-1): final states
          const int r0 = Bt(t + 1), nr = Bs - r0;
          if (nr > 0 && hT)
            RNN_TRY(copy_async(h, static_cast<char*>(hT) + ((size_t)v * BH + (size_t)r0 * H) * e, static_cast<const char*>(a.h_out) + (size_t)r0 * H * e, (size_t)nr * H * e, s));
          if (nr > 0 && cT && lstm)
            RNN_TRY(copy_async(h, cT + (size_t)v * BH + (size_t)r0 * H, a.c_out + (size_t)r0 * H, (size_t)nr * H * 4, s));
        }
      }
      // the top layer's output y[T][B][2H] = [h_forward(t), h_reverse(t)]
      if (l == L - 1) {
        RNN_TRY(copy2d_async(h, static_cast<char*>(y) + (size_t)dd * H * e, 2 * H * e, hseq + hslot(dd, 0) * BH * e, H * e, H * e, (size_t)T * B, s));
        // the reverse h sequence holds h0 rows where sequences start: y is 0 at idle positions
        if (dd == 1 && vl)
          for (int t = 0; t < T; ++t)
            if (Bt(t) < B)
              RNN_TRY(cu(cudaMemset2DAsync(static_cast<char*>(y) + ((size_t)t * B + Bt(t)) * 2 * H * e + H * e,
                                           2 * H * e, 0, H * e, (size_t)(B - Bt(t)), s)));
      }
    }
    if (side) RNN_TRY(join_streams(h, caller));
  }
  return RNN_OK;
}

int bwd_bidir(rnn_s* h, const void* dy, const void* dhT, const float* dcT, const char* PW, const float* c0, void* dx,
              void* dh0, float* dc0, char* R, char* W, void* ws, cudaStream_t s) {
  const rnn_desc_t& d = h->d;
  const int L = d.layers, T = d.T, B = d.B, H = d.hidden, GH = h->GH, mode = d.mode;
  const size_t e = h->elem, BH = (size_t)B * H, BGH = (size_t)B * GH;
  const bool lstm = d.cell == RNN_LSTM, gru = d.cell == RNN_GRU;
  const Remap none{0, 1, 1, 1};
  for (int v = 0; v < 2 * L; ++v)
    RNN_TRY(zero_async(h, W + h->wl[v].ctr, (size_t)h->ctr_count * 4, s));
  // variable lengths: rows 0 .. Bt[t]-1 run at time t; the gate gradients of
  // idle positions are never written, so they start at zero for the products
  // that read every row (dx, dW)
  const bool vl = h->varlen != 0;
  auto Bt = [&](int t) { return vl ? h->Bt[t] : (t < T ? B : 0); };
  if (vl)
    for (int v = 0; v < 2 * L; ++v) {
      RNN_TRY(zero_async(h, R + h->rl[v].dgx, (size_t)T * BGH * e, s));
      if (h->rl[v].dgh != h->rl[v].dgx) RNN_TRY(zero_async(h, R + h->rl[v].dgh, (size_t)T * BGH * e, s));
    }
  // the two halves of dy, each [T][B][H]
  for (int dd = 0; dd < 2; ++dd)
    RNN_TRY(copy2d_async(h, W + h->ws_dtop + (size_t)dd * T * BH * e, H * e, static_cast<const char*>(dy) + (size_t)dd * H * e, 2 * H * e, H * e, (size_t)T * B, s));
  cudaStream_t caller = s;
  const bool side = !(d.flags & RNN_FLAG_NO_WAVEFRONT);  // directions side by side
  for (int l = L - 1; l >= 0; --l) {
    if (side) RNN_TRY(fork_streams(h, caller));
    for (int dd = 0; dd < 2; ++dd) {
      const int v = 2 * l + dd;
      s = side ? h->streams[dd] : caller;
      const bool top = l == L - 1;
      const char* dyl = top ? W + h->ws_dtop + (size_t)dd * T * BH * e : W + h->wl[v].dyab;
      const size_t dy_es = top ? e : 4;
      float* carry = reinterpret_cast<float*>(W + h->wl[v].carry);
      char* hseq = R + h->rl[v].hseq;
      const float* c0v = c0 ? c0 + v * BH : nullptr;
      if (lstm || gru) {
        if (lstm && dcT) RNN_TRY(copy_async(h, carry, dcT + v * BH, BH * 4, s));
        else RNN_TRY(zero_async(h, carry, BH * 4, s));
      }
      // time of the k-th step of this direction's forward pass
      auto time_at = [&](int k) { return dd == 0 ? k : T - 1 - k; };
      auto args_for = [&](int k) {
        const int t = time_at(k), tp = dd == 0 ? t - 1 : t + 1;
        BwdStepArgs a;
        std::memset(&a, 0, sizeof(a));
        a.B = B;
        a.H = H;
        a.u = h->u;
        a.gates = reinterpret_cast<const float*>(R + h->rl[v].gates) + (size_t)t * BGH;
        a.c_s = lstm ? reinterpret_cast<const float*>(R + h->rl[v].c) + (size_t)t * BH : nullptr;
        a.c_sm1 = lstm ? (k > 0 ? reinterpret_cast<const float*>(R + h->rl[v].c) + (size_t)tp * BH : c0v) : nullptr;
        a.hn_s = gru ? reinterpret_cast<const float*>(R + h->rl[v].hn) + (size_t)t * BH : nullptr;
        a.h_sm1 = hseq + hslot(dd, tp) * BH * e;
        a.dy = dyl + (size_t)t * BH * dy_es;
        a.dy_f32 = top ? (mode == RNN_MODE_FP32) : 1;
        a.carry = carry;
        a.dGx = R + h->rl[v].dgx + (size_t)t * BGH * e;
        a.dGh = R + h->rl[v].dgh + (size_t)t * BGH * e;
        a.part = reinterpret_cast<float*>(W + h->wl[v].part);
        a.counters = reinterpret_cast<int*>(W + h->wl[v].ctr);
        a.cluster_splitk = 1;
        return a;
      };
      // the arguments of args_for moved down by r0 batch rows
      auto offset_rows = [&](BwdStepArgs x, int r0) {
        x.gates += (size_t)r0 * GH;
        if (x.c_s) x.c_s += (size_t)r0 * H;
        if (x.c_sm1) x.c_sm1 += (size_t)r0 * H;
        if (x.hn_s) x.hn_s += (size_t)r0 * H;
        if (x.h_sm1) x.h_sm1 = static_cast<const char*>(x.h_sm1) + (size_t)r0 * H * e;
        x.dy = static_cast<const char*>(x.dy) + (size_t)r0 * H * dy_es;
        x.carry += (size_t)r0 * H;
        x.dGx = static_cast<char*>(x.dGx) + (size_t)r0 * GH * e;
        x.dGh = static_cast<char*>(x.dGh) + (size_t)r0 * GH * e;
        return x;
      };
      auto point_args = [&](const BwdStepArgs& x, int k, int r0, int rows) {
        PointVArgs pv{};
        pv.B = rows;
        pv.H = H;
        pv.dy = x.dy;
        pv.dy_f32 = x.dy_f32;
        pv.gates = x.gates;
        pv.c_s = x.c_s;
        pv.c_sm1 = x.c_sm1;
        pv.carry = x.carry;
        pv.dc0 = (k == 0 && dc0 && lstm) ? dc0 + v * BH + (size_t)r0 * H : nullptr;
        pv.dGx = x.dGx;
        return pv;
      };
      Operand Bw{PW + h->pl[v].wh, H, 1, H, GH, 1};
      const char* dhTv = dhT ? static_cast<const char*>(dhT) + v * BH * e : nullptr;
      // the forward steps in reverse order.  Rows 0 .. Bn-1 take the product
      // of the gate gradients of the forward step after this one (time tn);
      // rows Bn .. Bs-1 start from dhT (forward: sequences ending at t)
      for (int k = T - 1; k >= 0; --k) {
        const int t = time_at(k), tn = dd == 0 ? t + 1 : t - 1;
        const int Bs = Bt(t);
        if (Bs == 0) continue;
        const int Bn = k == T - 1 ? 0 : (dd == 0 ? Bt(t + 1) : Bs);
        if (Bn > 0) {
          BwdStepArgs a = args_for(k);
          a.B = Bn;
          Operand A{R + h->rl[v].dgh + (size_t)tn * BGH * e, GH, 0, Bn, GH};
          Launch Lk = mk(h, s, ws, "bwd_step");
          if (h->tstep) {
            PointVArgs pv = point_args(a, k, 0, Bn);
            const int bnn = Bn > 128 ? 256 : Bn > 64 ? 128 : 64;
            int sp = h->bwd_splits;
            while (sp > 1 && bnn % (16 * sp)) sp /= 2;
            const bool fuse = h->bwd_fuse && bnn == 256 && sp == 4;
            float* dhb = reinterpret_cast<float*>(W + h->wl[v].dh);
            RNN_TRY(bwd_dh_t(Lk, Bw, A, Bn, H, h->G, bnn, sp, dhb, nullptr, 0,
                             reinterpret_cast<float*>(W + h->wl[v].part), a.gates, a.c_s, a.c_sm1,
                             fuse ? &pv : nullptr));
            if (!fuse) {
              pv.dh = dhb;
              Launch Lp = mk(h, s, ws, "bwd_point");
              RNN_TRY(bwd_point_v(Lp, d.cell, pv));
            }
          } else {
            RNN_TRY(bwd_step(Lk, mode, d.cell, A, Bw, h->bwd_bn, h->bwd_splits, a));
          }
        }
        if (Bs > Bn) {
          BwdStepArgs ar = offset_rows(args_for(k), Bn);
          ar.B = Bs - Bn;
          const char* dh_init = dhTv ? dhTv + (size_t)Bn * H * e : nullptr;
          Launch Lp = mk(h, s, ws, "bwd_point");
          if (h->tstep) {
            PointVArgs pv = point_args(ar, k, Bn, Bs - Bn);
            pv.dh_init = dh_init;
            RNN_TRY(bwd_point_v(Lp, d.cell, pv));
          } else {
            RNN_TRY(bwd_point(Lp, mode, d.cell, ar, dh_init));
          }
        }
        // reverse direction with variable lengths: rows Bt[t+1] .. Bs-1 began
        // their sweep at t, so their dh0 and dc0 are due now
        if (dd == 1 && vl) {
          const int r0 = Bt(t + 1), nr = Bs - r0;
          if (nr > 0 && dh0) {
            BwdStepArgs a = offset_rows(args_for(k), r0);
            a.B = nr;
            a.final_ = 1;
            a.dh0 = static_cast<char*>(dh0) + ((size_t)v * BH + (size_t)r0 * H) * e;
            a.dc0 = nullptr;
            Operand A{R + h->rl[v].dgh + ((size_t)t * BGH + (size_t)r0 * GH) * e, GH, 0, nr, GH};
            Launch Lk = mk(h, s, ws, "bwd_step");
            if (h->tstep) {
              const int bnn = nr > 128 ? 256 : nr > 64 ? 128 : 64;
              int sp = h->bwd_splits;
              while (sp > 1 && bnn % (16 * sp)) sp /= 2;
              RNN_TRY(bwd_dh_t(Lk, Bw, A, nr, H, h->G, bnn, sp, nullptr, a.dh0, 1,
                               reinterpret_cast<float*>(W + h->wl[v].part)));
            } else {
              RNN_TRY(bwd_step(Lk, mode, d.cell, A, Bw, h->bwd_bn, h->bwd_splits, a));
            }
          }
          // the carry out of the sequence's first step is its dc0
          if (nr > 0 && dc0 && lstm)
            RNN_TRY(copy_async(h, dc0 + v * BH + (size_t)r0 * H, carry + (size_t)r0 * H, (size_t)nr * H * 4, s));
        }
      }
      if (!(dd == 1 && vl) && (dh0 || (dc0 && lstm))) {
        BwdStepArgs a = args_for(0);
        a.final_ = 1;
        a.dh0 = dh0 ? static_cast<char*>(dh0) + v * BH * e : nullptr;
        a.dc0 = (dc0 && lstm) ? dc0 + v * BH : nullptr;
        Operand A{R + h->rl[v].dgh + (size_t)time_at(0) * BGH * e, GH, 0, B, GH};
        Launch Lk = mk(h, s, ws, "bwd_step");
        if (h->tstep) {
          // dc0 came out of the first step's pointwise kernel
          if (dh0)
            RNN_TRY(bwd_dh_t(Lk, Bw, A, B, H, h->G, h->bwd_bn, h->bwd_splits, nullptr, a.dh0, 1,
                             reinterpret_cast<float*>(W + h->wl[v].part)));
        } else {
          RNN_TRY(bwd_step(Lk, mode, d.cell, A, Bw, h->bwd_bn, h->bwd_splits, a));
        }
      }
    }
    if (side) RNN_TRY(join_streams(h, caller));
    // gradient of the layer input: dGx W_x, both directions summed (on the
    // caller's stream, one product after the other)
    s = caller;
    for (int dd = 0; dd < 2; ++dd) {
      const int v = 2 * l + dd;
      Operand A{R + h->rl[v].dgx, GH, 0, T * B, GH};
      if (l > 0) {
        // into the gradients from above of the two directions of layer l - 1
        for (int q = 0; q < 2; ++q) {
          Operand Bx{PW + h->pl[v].wx + (size_t)q * H * e, 2 * H, 1, H, GH, 1};
          Launch Lk = mk(h, s, ws, "dx_gemm");
          RNN_TRY(gemm_f32(Lk, mode, A, Bx, T * B, H, GH, reinterpret_cast<float*>(W + h->wl[2 * (l - 1) + q].dyab), H,
                           nullptr, dd, none, 0));
        }
      } else if (dx) {
        const int In = d.input;
        Operand Bx{PW + h->pl[v].wx, In, 1, In, GH, 1};
        Launch Lk = mk(h, s, ws, "dx_gemm");
        if (mode == RNN_MODE_FP32) {
          RNN_TRY(gemm_f32(Lk, mode, A, Bx, T * B, In, GH, static_cast<float*>(dx), In, nullptr, dd, none, 0));
        } else {
          float* acc = reinterpret_cast<float*>(W + h->ws_dxacc);
          RNN_TRY(gemm_f32(Lk, mode, A, Bx, T * B, In, GH, acc, In, nullptr, dd, none, 0));
          if (dd == 1) {
            Launch Lc = mk(h, s, ws, "cast");
            RNN_TRY(cast_bf16(Lc, acc, dx, (size_t)T * B * In));
          }
        }
      }
    }
  }
  return RNN_OK;
}

int wgrad_bidir(rnn_s* h, const void* x, const char* R, float* dw, int accumulate, void* ws, cudaStream_t s) {
  const rnn_desc_t& d = h->d;
  const int L = d.layers, T = d.T, B = d.B, H = d.hidden, G = h->G, GH = h->GH, mode = d.mode;
  const size_t e = h->elem, BH = (size_t)B * H;
  const int TB = T * B;
  const Remap rm{1, G, h->u, H};
  for (int v = 0; v < 2 * L; ++v) {
    const int l = v / 2, dd = v % 2;
    Operand dgx{R + h->rl[v].dgx, GH, 1, GH, TB};
    Operand dgh{R + h->rl[v].dgh, GH, 1, GH, TB};
    Launch Lk = mk(h, s, ws, "dw_gemm");
    if (l == 0) {
      const int In = d.input;
      Operand X{x, In, 1, In, TB};
      RNN_TRY(gemm_f32(Lk, mode, dgx, X, GH, In, TB, dw + h->ul[v].wx, In, nullptr, accumulate, rm, 0));
    } else {
      // the two halves of dW_x: inputs from the two directions of layer l - 1
      for (int q = 0; q < 2; ++q) {
        Operand X{R + h->rl[2 * (l - 1) + q].hseq + hslot(q, 0) * BH * e, H, 1, H, TB};
        RNN_TRY(gemm_f32(Lk, mode, dgx, X, GH, H, TB, dw + h->ul[v].wx + (size_t)q * H, 2 * H, nullptr, accumulate, rm,
                         0));
      }
    }
    // h before the step at time t: slot t (forward) or t + 1 (reverse)
    Operand Hp{R + h->rl[v].hseq + (size_t)dd * BH * e, H, 1, H, TB};
    RNN_TRY(gemm_f32(Lk, mode, dgh, Hp, GH, H, TB, dw + h->ul[v].wh, H, nullptr, accumulate, rm, 0));
    Launch Lb = mk(h, s, ws, "bias_grad");
    RNN_TRY(bias_grad(Lb, mode, d.cell, H, h->u, TB, R + h->rl[v].dgx, R + h->rl[v].dgh, dw + h->ul[v].bx,
                      dw + h->ul[v].bh, accumulate, reinterpret_cast<float*>(static_cast<char*>(ws) + h->ws_bias),
                      h->bias_slices));
  }
  return RNN_OK;
}

}  // namespace

// ======================================================================= C ABI
extern "C" {

const char* rnn_strerror(int code) {
  switch (code) {
    case RNN_OK: return "ok";
    case RNN_ERR_INVALID_ARG: return "invalid argument";
    case RNN_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case RNN_ERR_LAUNCH: return "kernel launch failed (resources or co-residency)";
    case RNN_ERR_CUDA: return "CUDA runtime error";
    case RNN_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case RNN_ERR_NOMEM: return "host allocation failed";
    default: return "unknown error";
  }
}

int rnn_create(const rnn_desc_t* desc, rnn_handle_t* out) {
  if (!desc || !out) return RNN_ERR_INVALID_ARG;
  *out = nullptr;
  const rnn_desc_t& d = *desc;
  if (d.cell < 0 || d.cell > 3 || d.mode < 0 || d.mode > 1 || d.layers < 1 || d.T < 1 || d.B < 1 ||
      d.input < 1 || d.hidden < 1)
    return RNN_ERR_INVALID_ARG;
  if ((d.flags & RNN_FLAG_FORCE_STREAMING) && (d.flags & RNN_FLAG_FORCE_PERSISTENT)) return RNN_ERR_INVALID_ARG;
  rnn_s* h = new (std::nothrow) rnn_s();
  if (!h) return RNN_ERR_NOMEM;
  h->d = d;
  int dev = 0, n = 0;
  if (cudaGetDeviceCount(&n) == cudaSuccess && n > 0 && cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
      h->num_sms = prop.multiProcessorCount;
      h->have_device = 1;
    }
  } else {
    cudaGetLastError();  // no device: host-side planning still works
  }
  int rc = plan_and_layout(h);
  if (rc != RNN_OK) {
    delete h;
    return rc;
  }
  h->prof = new (std::nothrow) Profiler();
  *out = h;
  return RNN_OK;
}

int rnn_destroy(rnn_handle_t h) {
  if (!h) return RNN_ERR_INVALID_ARG;
  if (!h->streams.empty()) {
    for (auto s : h->streams) cudaStreamSynchronize(s);
    for (auto s : h->streams) cudaStreamDestroy(s);
    for (auto e : h->ev) cudaEventDestroy(e);
    for (auto e : h->ev_join) cudaEventDestroy(e);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  }
  if (!h->graphs.empty()) cudaDeviceSynchronize();
  for (auto& g : h->graphs) {
    cudaGraphExecDestroy(g.exec);
    for (auto& r : g.prof) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
  }
  if (h->cap) cudaStreamDestroy(h->cap);
  delete h->prof;
  delete h;
  return RNN_OK;
}

namespace {
// drop every cached launch graph (the launch sequence changed)
void clear_graphs(rnn_s* h) {
  if (!h->graphs.empty()) cudaDeviceSynchronize();
  for (auto& g : h->graphs) {
    cudaGraphExecDestroy(g.exec);
    for (auto& r : g.prof) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
  }
  h->graphs.clear();
  h->seen.clear();
  h->no_graph.clear();
}
}  // namespace

int rnn_set_lengths(rnn_handle_t h, const int* lens) {
  if (!h) return RNN_ERR_INVALID_ARG;
  const int T = h->d.T, B = h->d.B;
  if (lens) {
    for (int b = 0; b < B; ++b)
      if (lens[b] < 1 || lens[b] > T || (b > 0 && lens[b] > lens[b - 1])) return RNN_ERR_INVALID_ARG;
  }
  clear_graphs(h);
  h->varlen = (lens && lens[B - 1] < T) ? 1 : 0;
  h->Bt.assign(T + 1, 0);
  for (int t = 0; t < T; ++t) {
    int n = 0;
    while (n < B && (!lens || lens[n] > t)) ++n;
    h->Bt[t] = n;
  }
  // the persistent recurrence runs all T steps of every sequence: step
  // launches take over (the packing unit it was planned with serves them)
  h->persist = h->varlen ? 0 : h->persist_plan;
  h->stack = h->varlen ? 0 : h->stack_plan;
  h->stackb = h->varlen ? 0 : h->stackb_plan;
  return RNN_OK;
}

int rnn_get_sizes(rnn_handle_t h, size_t* user_weight_bytes, size_t* packed_weight_bytes, size_t* reserve_bytes,
                  size_t* workspace_bytes) {
  if (!h) return RNN_ERR_INVALID_ARG;
  if (user_weight_bytes) *user_weight_bytes = h->user_w_bytes;
  if (packed_weight_bytes) *packed_weight_bytes = h->packed_bytes;
  if (reserve_bytes) *reserve_bytes = h->reserve_bytes;
  if (workspace_bytes) *workspace_bytes = h->ws_bytes;
  return RNN_OK;
}

int rnn_describe(rnn_handle_t h, char* buf, size_t len) {
  if (!h || !buf || len == 0) return RNN_ERR_INVALID_ARG;
  const char* cell = h->d.cell == RNN_LSTM ? "lstm" : h->d.cell == RNN_GRU ? "gru" : h->d.cell == RNN_RELU ? "relu" : "tanh";
  // layer groups of the stacked forward, "first+count" each
  char groups[128] = "-", bgroups[128] = "-";
  auto list = [](char* out, size_t len, const std::vector<std::pair<int, int>>& gs) {
    size_t n = 0;
    for (size_t i = 0; i < gs.size() && n + 16 < len; ++i)
      n += (size_t)snprintf(out + n, len - n, "%s%d+%d", i ? "," : "", gs[i].first, gs[i].second);
  };
  if (h->stack) list(groups, sizeof(groups), h->stack_groups);
  if (h->stackb) list(bgroups, sizeof(bgroups), h->stackb_groups);
  if (h->stackb && h->stackb_rec) strncat(bgroups, "r", sizeof(bgroups) - strlen(bgroups) - 1);
  snprintf(buf, len,
           "cell=%s mode=%s L=%d T=%d B=%d I=%d H=%d G=%d u=%d recurrence=%s engine=%s wavefront=%d "
           "chunk=%d nchunks=%d bwd_bn=%d bwd_splits=%d sms=%d transposed=%d fused_point=%d "
           "persist_cluster=%d directions=%d fp8_stash=%d stack_groups=%s stack_bwd_groups=%s slim_step=%d "
           "step_chunks=%d",
           cell, h->d.mode ? "bf16" : "fp32", h->d.layers, h->d.T, h->d.B, h->d.input, h->d.hidden, h->G, h->u,
           h->persist ? "persistent" : h->stack ? "stacked" : "streaming", h->d.mode ? "tcgen05" : "ffma",
           h->wavefront, h->chunk, h->nch, h->bwd_bn, h->bwd_splits, h->num_sms, h->tstep, h->bwd_fuse,
           h->persist ? h->persist_cl : 0, h->D, h->persist8, groups, bgroups, h->slim_step,
           h->step_chunks);
  return RNN_OK;
}

unsigned long long rnn_launch_count(void) { return g_launches.load(); }

int rnn_pack_weights(rnn_handle_t h, const void* w_user, void* w_packed, cudaStream_t stream) {
  if (!h || !w_user || !w_packed) return RNN_ERR_INVALID_ARG;
  if (!aligned16(w_user) || !aligned16(w_packed)) return RNN_ERR_INVALID_ARG;
  RNN_TRY(ensure_runtime(h));
  const char* U = static_cast<const char*>(w_user);
  char* P = static_cast<char*>(w_packed);
  const size_t e = h->elem;
  for (int l = 0; l < h->V(); ++l) {
    Launch L = mk(h, stream, nullptr, "pack");
    RNN_TRY(pack_layer(L, h->d.mode, h->d.cell, h->d.hidden, h->In(l / h->D), h->u, U + h->ul[l].wx * e,
                       U + h->ul[l].wh * e, U + h->ul[l].bx * e, U + h->ul[l].bh * e, P + h->pl[l].wx,
                       P + h->pl[l].wh, reinterpret_cast<float*>(P + h->pl[l].bias),
                       reinterpret_cast<float*>(P + h->pl[l].bias_hn)));
    if (h->d.flags & RNN_FLAG_FP8_STASH) {
      // the e4m3 stash of the packed W_h rows with one scale per row
      Launch Lq = mk(h, stream, nullptr, "pack");
      RNN_TRY(quant_rows_e4m3(Lq, P + h->pl[l].wh, h->GH, h->d.hidden, reinterpret_cast<uint8_t*>(P + h->pl[l].wh8),
                              reinterpret_cast<float*>(P + h->pl[l].wsc)));
    }
  }
  return RNN_OK;
}

int rnn_fwd(rnn_handle_t h, const void* x, const void* h0, const float* c0, const void* w_packed, void* y,
            void* hT, float* cT, void* reserve, void* ws, cudaStream_t stream) {
  if (!h || !x || !w_packed || !y || !ws) return RNN_ERR_INVALID_ARG;
  for (const void* p : {x, h0, (const void*)c0, w_packed, (const void*)y, (const void*)hT, (const void*)cT,
                        (const void*)reserve, (const void*)ws})
    if (!aligned16(p)) return RNN_ERR_INVALID_ARG;
  RNN_TRY(ensure_runtime(h));
  const std::vector<uintptr_t> key = {1, (uintptr_t)x, (uintptr_t)h0, (uintptr_t)c0, (uintptr_t)w_packed, (uintptr_t)y, (uintptr_t)hT, (uintptr_t)cT, (uintptr_t)reserve, (uintptr_t)ws};
  auto issue = [&](cudaStream_t stream) -> int {
    const rnn_desc_t& d = h->d;
    const int L = d.layers, T = d.T, B = d.B, H = d.hidden, G = h->G, GH = h->GH, mode = d.mode;
    const size_t e = h->elem, BH = (size_t)B * H, BGH = (size_t)B * GH;
    const bool train = reserve != nullptr;
    const bool lstm = d.cell == RNN_LSTM, gru = d.cell == RNN_GRU;
    char* R = static_cast<char*>(reserve);
    char* W = static_cast<char*>(ws);
    const char* PW = static_cast<const char*>(w_packed);
    (void)G;
    if (h->D == 2) return fwd_bidir(h, x, h0, c0, PW, y, hT, cT, R, W, ws, stream);
    // inference with the fp8 stash: the persistent recurrence on e4m3 W_h,
    // layer after layer (no wavefront)
    const bool p8 = !train && h->persist8 && !h->varlen;
    if (!p8 && h->stack && !h->varlen) return fwd_stack(h, x, h0, c0, PW, y, hT, cT, R, W, ws, stream);
    const bool pers = p8 || h->persist;
    const int wf = p8 ? 0 : h->wavefront;
    const int nch = p8 ? 1 : h->nch;
    const int chunk = p8 ? T : h->chunk;

    if (h->varlen) {
      // rows past a sequence's end are never written by the steps: y reads 0
      // there, and the h sequences the weight gradients and the next layer
      // read hold zeros instead of stale memory
      RNN_TRY(zero_async(h, y, (size_t)T * BH * e, stream));
      for (int l = 0; l < L; ++l)
        RNN_TRY(zero_async(h, train ? R + h->rl[l].hseq : W + h->wl[l].hseq, (size_t)(T + 1) * BH * e, stream));
    }
    // several steps per launch: arrival counters per (layer, step), zeroed once per call
    const bool chunks = h->step_chunks && train && !pers && !h->varlen;
    unsigned int* step_cnt = reinterpret_cast<unsigned int*>(W + h->ws_arrive);
    if (chunks) RNN_TRY(zero_async(h, step_cnt, (size_t)L * T * 4, stream));
    if (wf) RNN_TRY(fork_streams(h, stream));
    const int nd = wf ? (L + nch - 1) : 1;
    for (int dg = 0; dg < nd; ++dg) {
      for (int l = 0; l < L; ++l) {
        for (int c = 0; c < nch; ++c) {
          if (wf && l + c != dg) continue;
          cudaStream_t s = wf ? h->streams[l] : stream;
          const int t0 = c * chunk, t1 = std::min(T, t0 + chunk);
          char* hseq = train ? R + h->rl[l].hseq : W + h->wl[l].hseq;
          float* P = reinterpret_cast<float*>(train ? R + h->rl[l].gates : W + h->wl[l].P);
          if (c == 0) {
            if (h0) RNN_TRY(copy_async(h, hseq, static_cast<const char*>(h0) + l * BH * e, BH * e, s));
            else RNN_TRY(zero_async(h, hseq, BH * e, s));
          }
          if (wf && l > 0) RNN_TRY(cu(cudaStreamWaitEvent(s, h->ev[(size_t)(l - 1) * nch + c], 0)));
          // input projection (layer 0: all T at once)
          if (l > 0 || c == 0) {
            const int r0 = l == 0 ? 0 : t0, r1 = l == 0 ? T : t1;
            const int In = h->In(l);
            Operand A;
            A.ptr = l == 0 ? static_cast<const char*>(x) + (size_t)r0 * B * In * e
                           : static_cast<const char*>(train ? R + h->rl[l - 1].hseq : W + h->wl[l - 1].hseq) +
                                 (size_t)(r0 + 1) * BH * e;
            A.ld = In;
            A.mn_major = 0;
            A.mn_ext = (r1 - r0) * B;
            A.k_ext = In;
            Operand Bw{PW + h->pl[l].wx, In, 0, GH, In, 1};
            Remap none{0, 1, 1, 1};
            Launch Lk = mk(h, s, ws, "input_proj_gemm");
            RNN_TRY(gemm_f32(Lk, mode, A, Bw, (r1 - r0) * B, GH, In, P + (size_t)r0 * BGH, GH,
                             reinterpret_cast<const float*>(PW + h->pl[l].bias), 0, none, 0));
          }
          // persistent recurrence: all T steps of the layer in one launch
          if (pers) {
            unsigned int* arrive = reinterpret_cast<unsigned int*>(W + h->ws_arrive);
            if (pa_cluster(h, p8)) RNN_TRY(zero_async(h, W + h->ws_hx, (size_t)8 * B * H, s));
            else RNN_TRY(zero_async(h, arrive, (size_t)T * 4, s));
            PersistArgs pa{};
            pa.arrive = arrive;
            pa.cluster = p8 ? h->persist8_cl : h->persist_cl;
            pa.cluster_sync = (d.flags & RNN_FLAG_PERSIST_CLUSTER_SYNC) ? 1 : 0;
            pa.Wh8 = p8 ? reinterpret_cast<const uint8_t*>(PW + h->pl[l].wh8) : nullptr;
            pa.wscale = p8 ? reinterpret_cast<const float*>(PW + h->pl[l].wsc) : nullptr;
            pa.hx = reinterpret_cast<uint64_t*>(W + h->ws_hx);
            pa.T = T;
            pa.B = B;
            pa.H = H;
            pa.u_pack = h->u;
            pa.Wh = reinterpret_cast<const __nv_bfloat16*>(PW + h->pl[l].wh);
            pa.P = P;
            pa.gates_out = train ? P : nullptr;
            pa.bias_hn = reinterpret_cast<const float*>(PW + h->pl[l].bias_hn);
            pa.c0 = (lstm && c0) ? c0 + l * BH : nullptr;
            pa.c_out = (train && lstm) ? reinterpret_cast<float*>(R + h->rl[l].c) : nullptr;
            pa.hn_out = (train && gru) ? reinterpret_cast<float*>(R + h->rl[l].hn) : nullptr;
            pa.hseq = reinterpret_cast<__nv_bfloat16*>(hseq);
            pa.y = l == L - 1 ? static_cast<__nv_bfloat16*>(y) : nullptr;
            pa.hT = hT ? reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(hT) + (size_t)l * BH * e) : nullptr;
            pa.cT = (cT && lstm) ? cT + (size_t)l * BH : nullptr;
            pa.err = reinterpret_cast<int*>(W + h->ws_err);
            pa.limit_ns = h->limit_ns;
            pa.test_skip_publish = (d.flags & RNN_FLAG_TEST_SKIP_PUBLISH) ? 1 : 0;
            Launch Lk = mk(h, s, ws, "persist_fwd");
            RNN_TRY(persist_fwd(Lk, d.cell, pa));
            continue;
          }
          // recurrent steps of the chunk (with variable lengths only the
          // Bt[t] sequences still running, rows 0 .. Bt[t]-1)
          for (int t = t0; t < t1; ++t) {
            const int Bs = h->varlen ? h->Bt[t] : B;
            if (Bs == 0) continue;
            // the chunk's steps from t on in one launch (t = 0 reads c0 and runs alone)
            const int ns = (chunks && t > 0) ? t1 - t : 1;
            const int tl = t + ns - 1;
            FwdStepArgs a;
            a.B = Bs;
            a.H = H;
            a.u = h->u;
            a.P = P + (size_t)t * BGH;
            a.write_gates = train ? 1 : 0;
            a.bias_hn = reinterpret_cast<const float*>(PW + h->pl[l].bias_hn);
            auto cbuf = [&](int tt) -> float* {
              return train ? reinterpret_cast<float*>(R + h->rl[l].c) + (size_t)tt * BH
                           : reinterpret_cast<float*>(W + h->wl[l].c2) + (size_t)(tt & 1) * BH;
            };
            a.c_prev = lstm ? (t == 0 ? (c0 ? c0 + l * BH : nullptr) : cbuf(t - 1)) : nullptr;
            a.c_out = lstm ? cbuf(t) : nullptr;
            a.h_prev = hseq + (size_t)t * BH * e;
            a.h_out = hseq + (size_t)(t + 1) * BH * e;
            a.y = l == L - 1 ? static_cast<char*>(y) + (size_t)t * BH * e : nullptr;
            a.hT = (!h->varlen && tl == T - 1 && hT) ? static_cast<char*>(hT) + (size_t)l * BH * e : nullptr;
            a.cT = (!h->varlen && tl == T - 1 && cT && lstm) ? cT + (size_t)l * BH : nullptr;
            a.hn_out = (train && gru) ? reinterpret_cast<float*>(R + h->rl[l].hn) + (size_t)t * BH : nullptr;
            a.slim = h->slim_step;
            a.steps = ns;
            a.hT_step = T - 1 - t;
            a.step_cnt = ns > 1 ? step_cnt + (size_t)l * T + t : nullptr;
            Operand A{hseq + (size_t)t * BH * e, H, 0, Bs, H};
            Operand Bw{PW + h->pl[l].wh, H, 0, GH, H, 1};
            Launch Lk = mk(h, s, ws, "fwd_step");
            if (h->tstep) RNN_TRY(fwd_step_t(Lk, d.cell, Bw, A, a));
            else RNN_TRY(fwd_step(Lk, mode, d.cell, A, Bw, a));
            if (h->varlen) {
              // sequences ending at step t (rows Bt[t+1] .. Bt[t]-1): final states
              const int r0 = h->Bt[t + 1], nr = Bs - r0;
              if (nr > 0 && hT)
                RNN_TRY(copy_async(h, static_cast<char*>(hT) + ((size_t)l * BH + (size_t)r0 * H) * e, static_cast<const char*>(a.h_out) + (size_t)r0 * H * e, (size_t)nr * H * e, s));
              if (nr > 0 && cT && lstm)
                RNN_TRY(copy_async(h, cT + (size_t)l * BH + (size_t)r0 * H, a.c_out + (size_t)r0 * H, (size_t)nr * H * 4, s));
            }
            t = tl;
          }
          if (wf) RNN_TRY(cu(cudaEventRecord(h->ev[(size_t)l * nch + c], s)));
        }
      }
    }
    if (wf) RNN_TRY(join_streams(h, stream));
    return RNN_OK;
  };
  return run_graphed(h, stream, key, issue);
}

int rnn_bwd_data(rnn_handle_t h, const void* dy, const void* dhT, const float* dcT, const void* w_packed,
                 const void* h0, const float* c0, void* dx, void* dh0, float* dc0, void* reserve, void* ws,
                 cudaStream_t stream) {
  if (!h || !dy || !w_packed || !reserve || !ws) return RNN_ERR_INVALID_ARG;
  for (const void* p : {dy, dhT, (const void*)dcT, w_packed, h0, (const void*)c0, (const void*)dx,
                        (const void*)dh0, (const void*)dc0, (const void*)reserve, (const void*)ws})
    if (!aligned16(p)) return RNN_ERR_INVALID_ARG;
  (void)h0;
  RNN_TRY(ensure_runtime(h));
  const std::vector<uintptr_t> key = {2, (uintptr_t)dy, (uintptr_t)dhT, (uintptr_t)dcT, (uintptr_t)w_packed, (uintptr_t)h0, (uintptr_t)c0, (uintptr_t)dx, (uintptr_t)dh0, (uintptr_t)dc0, (uintptr_t)reserve, (uintptr_t)ws};
  auto issue = [&](cudaStream_t stream) -> int {
    const rnn_desc_t& d = h->d;
    const int L = d.layers, T = d.T, B = d.B, H = d.hidden, GH = h->GH, mode = d.mode;
    const size_t e = h->elem, BH = (size_t)B * H, BGH = (size_t)B * GH;
    const bool lstm = d.cell == RNN_LSTM, gru = d.cell == RNN_GRU;
    char* R = static_cast<char*>(reserve);
    char* W = static_cast<char*>(ws);
    const char* PW = static_cast<const char*>(w_packed);
    if (h->D == 2) return bwd_bidir(h, dy, dhT, dcT, PW, c0, dx, dh0, dc0, R, W, ws, stream);
    if (h->stackb && !h->varlen) return bwd_stack(h, dy, dhT, dcT, PW, c0, dx, dh0, dc0, R, W, ws, stream);

    for (int l = 0; l < L; ++l)
      RNN_TRY(zero_async(h, W + h->wl[l].ctr, (size_t)h->ctr_count * 4, stream));
    if (h->varlen) {
      // gate gradients of finished sequences are never written: zero, so that
      // the products that read every row (dx, dW, the next step) see zeros
      for (int l = 0; l < L; ++l) {
        RNN_TRY(zero_async(h, R + h->rl[l].dgx, (size_t)T * BGH * e, stream));
        if (h->rl[l].dgh != h->rl[l].dgx)
          RNN_TRY(zero_async(h, R + h->rl[l].dgh, (size_t)T * BGH * e, stream));
      }
    }
    if (h->wavefront) RNN_TRY(fork_streams(h, stream));
    const int nd = h->wavefront ? (L + h->nch - 1) : 1;
    for (int dg = 0; dg < nd; ++dg) {
      for (int li = 0; li < L; ++li) {
        const int l = L - 1 - li;
        for (int rc = 0; rc < h->nch; ++rc) {
          if (h->wavefront && li + rc != dg) continue;
          cudaStream_t s = h->wavefront ? h->streams[l] : stream;
          const int t1 = T - rc * h->chunk, t0 = std::max(0, t1 - h->chunk);
          if (h->wavefront && l < L - 1) RNN_TRY(cu(cudaStreamWaitEvent(s, h->ev[(size_t)(l + 1) * h->nch + rc], 0)));
          const bool top = l == L - 1;
          const char* dyl = top ? static_cast<const char*>(dy) : W + h->wl[l].dyab;
          const size_t dy_es = top ? e : 4;
          float* carry = reinterpret_cast<float*>(W + h->wl[l].carry);
          char* hseq = R + h->rl[l].hseq;
          const float* c0l = c0 ? c0 + l * BH : nullptr;
          if (rc == 0 && (lstm || gru)) {
            if (lstm && dcT) RNN_TRY(copy_async(h, carry, dcT + l * BH, BH * 4, s));
            else RNN_TRY(zero_async(h, carry, BH * 4, s));
          }
          auto args_for = [&](int st) {
            BwdStepArgs a;
            std::memset(&a, 0, sizeof(a));
            a.B = B;
            a.H = H;
            a.u = h->u;
            a.gates = reinterpret_cast<const float*>(R + h->rl[l].gates) + (size_t)st * BGH;
            a.c_s = lstm ? reinterpret_cast<const float*>(R + h->rl[l].c) + (size_t)st * BH : nullptr;
            a.c_sm1 = lstm ? (st > 0 ? reinterpret_cast<const float*>(R + h->rl[l].c) + (size_t)(st - 1) * BH : c0l)
                           : nullptr;
            a.hn_s = gru ? reinterpret_cast<const float*>(R + h->rl[l].hn) + (size_t)st * BH : nullptr;
            a.h_sm1 = hseq + (size_t)st * BH * e;
            a.dy = dyl + (size_t)st * BH * dy_es;
            a.dy_f32 = top ? (mode == RNN_MODE_FP32) : 1;
            a.carry = carry;
            a.dGx = R + h->rl[l].dgx + (size_t)st * BGH * e;
            a.dGh = R + h->rl[l].dgh + (size_t)st * BGH * e;
            a.part = reinterpret_cast<float*>(W + h->wl[l].part);
            a.counters = reinterpret_cast<int*>(W + h->wl[l].ctr);
            a.cluster_splitk = 1;
            return a;
          };
          Operand Bw{PW + h->pl[l].wh, H, 1, H, GH, 1};
          // the arguments of args_for moved down by r0 batch rows
          auto offset_rows = [&](BwdStepArgs x, int r0) {
            x.gates += (size_t)r0 * GH;
            if (x.c_s) x.c_s += (size_t)r0 * H;
            if (x.c_sm1) x.c_sm1 += (size_t)r0 * H;
            if (x.hn_s) x.hn_s += (size_t)r0 * H;
            if (x.h_sm1) x.h_sm1 = static_cast<const char*>(x.h_sm1) + (size_t)r0 * H * e;
            x.dy = static_cast<const char*>(x.dy) + (size_t)r0 * H * dy_es;
            x.carry += (size_t)r0 * H;
            x.dGx = static_cast<char*>(x.dGx) + (size_t)r0 * GH * e;
            x.dGh = static_cast<char*>(x.dGh) + (size_t)r0 * GH * e;
            return x;
          };
          auto point_args = [&](const BwdStepArgs& x, int st, int r0, int rows) {
            PointVArgs pv{};
            pv.B = rows;
            pv.H = H;
            pv.dy = x.dy;
            pv.dy_f32 = x.dy_f32;
            pv.gates = x.gates;
            pv.c_s = x.c_s;
            pv.c_sm1 = x.c_sm1;
            pv.carry = x.carry;
            pv.dc0 = (st == 0 && dc0 && lstm) ? dc0 + l * BH + (size_t)r0 * H : nullptr;
            pv.dGx = x.dGx;
            return pv;
          };
          for (int st = t1 - 1; st >= t0; --st) {
            // rows 0 .. Bn-1 were running at st+1 (their dh has a recurrent
            // part); rows Bn .. Bs-1 end at st (their dh starts from dhT)
            const int Bs = h->varlen ? h->Bt[st] : B;
            const int Bn = st == T - 1 ? 0 : (h->varlen ? h->Bt[st + 1] : B);
            const char* dhTl = dhT ? static_cast<const char*>(dhT) + l * BH * e : nullptr;
            BwdStepArgs a = args_for(st);
            if (Bn > 0) {
              a.B = Bn;
              Operand A{R + h->rl[l].dgh + (size_t)(st + 1) * BGH * e, GH, 0, Bn, GH};
              Launch Lk = mk(h, s, ws, "bwd_step");
              if (h->tstep) {
                // transposed: the product writes dh_s (or runs the pointwise
                // step in its epilogue), else a pointwise kernel follows
                PointVArgs pv = point_args(a, st, 0, Bn);
                const int bnn = Bn > 128 ? 256 : Bn > 64 ? 128 : 64;
                int sp = h->bwd_splits;
                while (sp > 1 && bnn % (16 * sp)) sp /= 2;
                const bool fuse = h->bwd_fuse && bnn == 256 && sp == 4;
                float* dhb = reinterpret_cast<float*>(W + h->wl[l].dh);
                RNN_TRY(bwd_dh_t(Lk, Bw, A, Bn, H, h->G, bnn, sp, dhb, nullptr, 0,
                                 reinterpret_cast<float*>(W + h->wl[l].part), a.gates, a.c_s, a.c_sm1,
                                 fuse ? &pv : nullptr));
                if (!fuse) {
                  pv.dh = dhb;
                  Launch Lp = mk(h, s, ws, "bwd_point");
                  RNN_TRY(bwd_point_v(Lp, d.cell, pv));
                }
              } else {
                RNN_TRY(bwd_step(Lk, mode, d.cell, A, Bw, h->bwd_bn, h->bwd_splits, a));
              }
            }
            if (Bs > Bn) {
              BwdStepArgs ar = offset_rows(args_for(st), Bn);
              ar.B = Bs - Bn;
              const char* dh_init = dhTl ? dhTl + (size_t)Bn * H * e : nullptr;
              Launch Lp = mk(h, s, ws, "bwd_point");
              if (h->tstep) {
                PointVArgs pv = point_args(ar, st, Bn, Bs - Bn);
                pv.dh_init = dh_init;
                RNN_TRY(bwd_point_v(Lp, d.cell, pv));
              } else {
                RNN_TRY(bwd_point(Lp, mode, d.cell, ar, dh_init));
              }
            }
          }
          if (t0 == 0 && (dh0 || (dc0 && lstm))) {
            BwdStepArgs a = args_for(0);
            a.final_ = 1;
            a.dh0 = dh0 ? static_cast<char*>(dh0) + l * BH * e : nullptr;
            a.dc0 = (dc0 && lstm) ? dc0 + l * BH : nullptr;
            Operand A{R + h->rl[l].dgh, GH, 0, B, GH};
            Launch Lk = mk(h, s, ws, "bwd_step");
            if (h->tstep) {
              // dc0 came out of step 0's pointwise kernel
              if (dh0)
                RNN_TRY(bwd_dh_t(Lk, Bw, A, B, H, h->G, h->bwd_bn, h->bwd_splits, nullptr, a.dh0, 1,
                                 reinterpret_cast<float*>(W + h->wl[l].part)));
            } else {
              RNN_TRY(bwd_step(Lk, mode, d.cell, A, Bw, h->bwd_bn, h->bwd_splits, a));
            }
          }
          // gradient of this chunk's layer inputs: dGx W_x
          if (l > 0 || dx) {
            const int In = h->In(l);
            Operand A{R + h->rl[l].dgx + (size_t)t0 * BGH * e, GH, 0, (t1 - t0) * B, GH};
            Operand Bx{PW + h->pl[l].wx, In, 1, In, GH, 1};
            Launch Lk = mk(h, s, ws, "dx_gemm");
            if (l > 0) {
              Remap none{0, 1, 1, 1};
              RNN_TRY(gemm_f32(Lk, mode, A, Bx, (t1 - t0) * B, In, GH,
                               reinterpret_cast<float*>(W + h->wl[l - 1].dyab) + (size_t)t0 * BH, In, nullptr, 0, none,
                               0));
            } else {
              RNN_TRY(gemm_store(Lk, mode, A, Bx, (t1 - t0) * B, In, GH,
                                 static_cast<char*>(dx) + (size_t)t0 * B * In * e, In, 0));
            }
          }
          if (h->wavefront) RNN_TRY(cu(cudaEventRecord(h->ev[(size_t)l * h->nch + rc], s)));
        }
      }
    }
    if (h->wavefront) RNN_TRY(join_streams(h, stream));
    return RNN_OK;
  };
  return run_graphed(h, stream, key, issue);
}

int rnn_bwd_weights(rnn_handle_t h, const void* x, const void* h0, const void* reserve, float* dw, int accumulate,
                    void* ws, cudaStream_t stream) {
  if (!h || !x || !reserve || !dw || !ws) return RNN_ERR_INVALID_ARG;
  for (const void* p : {x, h0, reserve, (const void*)dw, (const void*)ws})
    if (!aligned16(p)) return RNN_ERR_INVALID_ARG;
  (void)h0;  // h_{-1} = h0 was stored in the reserve by the forward pass
  RNN_TRY(ensure_runtime(h));
  const std::vector<uintptr_t> key = {3, (uintptr_t)x, (uintptr_t)h0, (uintptr_t)reserve, (uintptr_t)dw, (uintptr_t)accumulate, (uintptr_t)ws};
  auto issue = [&](cudaStream_t stream) -> int {
    const rnn_desc_t& d = h->d;
    const int L = d.layers, T = d.T, B = d.B, H = d.hidden, G = h->G, GH = h->GH, mode = d.mode;
    const size_t e = h->elem, BH = (size_t)B * H;
    const char* R = static_cast<const char*>(reserve);
    const int TB = T * B;
    if (h->D == 2) return wgrad_bidir(h, x, R, dw, accumulate, ws, stream);
    // A weight-gradient product has about (G*H / 256) x (I_l / 256) tiles of
    // 256 x 256 on CTA pairs over K = T*B.  Where one fills the GPU, the
    // products run back to back on the caller's stream; where one would leave
    // most SMs idle (moderate widths), each layer's two products run on its
    // own stream, side by side with the other layers' (the outputs are
    // disjoint), each followed by its bias reduction (own scratch slice).
    const int tiles = ((GH + 255) / 256) * ((std::max(d.input, H) + 255) / 256);
    const bool side = L > 1 && 2 * tiles * 4 <= h->num_sms && !(d.flags & RNN_FLAG_PROFILE);
    if (side) RNN_TRY(fork_streams(h, stream));
    for (int l = 0; l < L; ++l) {
      const int In = h->In(l);
      Remap rm{1, G, h->u, H};
      Operand dgx{R + h->rl[l].dgx, GH, 1, GH, TB};
      Operand dgh{R + h->rl[l].dgh, GH, 1, GH, TB};
      Operand X = l == 0 ? Operand{x, In, 1, In, TB} : Operand{R + h->rl[l - 1].hseq + BH * e, H, 1, H, TB};
      Operand Hp{R + h->rl[l].hseq, H, 1, H, TB};
      Launch Lk = mk(h, side ? h->streams[l] : stream, ws, "dw_gemm");
      RNN_TRY(gemm_f32(Lk, mode, dgx, X, GH, In, TB, dw + h->ul[l].wx, In, nullptr, accumulate, rm, 0));
      RNN_TRY(gemm_f32(Lk, mode, dgh, Hp, GH, H, TB, dw + h->ul[l].wh, H, nullptr, accumulate, rm, 0));
    }
    for (int l = 0; l < L; ++l) {
      Launch Lb = mk(h, side ? h->streams[l] : stream, ws, "bias_grad");
      float* scratch = reinterpret_cast<float*>(static_cast<char*>(ws) + h->ws_bias) + (size_t)l * h->bias_slices * GH;
      RNN_TRY(bias_grad(Lb, mode, d.cell, H, h->u, TB, R + h->rl[l].dgx, R + h->rl[l].dgh, dw + h->ul[l].bx,
                        dw + h->ul[l].bh, accumulate, scratch, h->bias_slices));
    }
    if (side) RNN_TRY(join_streams(h, stream));
    return RNN_OK;
  };
  return run_graphed(h, stream, key, issue);
}

int rnn_sync_status(rnn_handle_t h, void* ws, cudaStream_t stream) {
  if (!h || !ws) return RNN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return RNN_ERR_CUDA;
  int word = 0;
  char* p = static_cast<char*>(ws) + h->ws_err;
  if (cudaMemcpy(&word, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return RNN_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return RNN_ERR_CUDA;
    return word == 3 /* DEV_BAD_CLUSTER (common.cuh) */ ? RNN_ERR_LAUNCH : RNN_ERR_TIMEOUT;
  }
  return RNN_OK;
}

int rnn_profile_query(rnn_handle_t h, int k, char* name, int* n_classes, unsigned long long* launches,
                      double* total_ms, int reset) {
  if (!h || !h->prof) return RNN_ERR_INVALID_ARG;
  if (h->have_device && cudaDeviceSynchronize() != cudaSuccess) return RNN_ERR_CUDA;
  Profiler& p = *h->prof;
  std::lock_guard<std::mutex> g(p.mu);
  p.settle();
  if (n_classes) *n_classes = (int)p.names.size();
  int rc = RNN_OK;
  if (k >= 0 && k < (int)p.names.size()) {
    if (name) {
      std::strncpy(name, p.names[k].c_str(), 31);
      name[31] = 0;
    }
    if (launches) *launches = p.launches[k];
    if (total_ms) *total_ms = p.total_ms[k];
  } else if (k >= 0) {
    rc = RNN_ERR_INVALID_ARG;
  }
  if (reset) {
    for (auto& v : p.launches) v = 0;
    for (auto& v : p.total_ms) v = 0.0;
  }
  return rc;
}

int rnn_gemm_bf16(int M, int N, int K, const void* A, long long lda, int a_mn_major, const void* B, long long ldb,
                  int b_mn_major, float* D, long long ldd, const float* bias, int accumulate, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !D) return RNN_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || ((lda * 2) & 15) || ((ldb * 2) & 15)) return RNN_ERR_INVALID_ARG;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return RNN_ERR_CUDA;
  Operand a{A, lda, a_mn_major ? 1 : 0, M, K};
  Operand b{B, ldb, b_mn_major ? 1 : 0, N, K};
  Launch L;
  L.stream = stream;
  L.err = nullptr;
  L.limit_ns = 2000000000ull;
  L.num_sms = prop.multiProcessorCount;
  L.prof = nullptr;
  L.name = "gemm";
  Remap none{0, 1, 1, 1};
  return gemm_f32(L, RNN_MODE_BF16, a, b, M, N, K, D, ldd, bias, accumulate, none, 0);
}

int rnn_quantize_e4m3_rows(int rows, int cols, const void* w, void* q, float* scale, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0 || !w || !q || !scale) return RNN_ERR_INVALID_ARG;
  Launch L;
  L.stream = stream;
  L.err = nullptr;
  L.limit_ns = 2000000000ull;
  L.num_sms = 0;
  L.prof = nullptr;
  L.name = "quant";
  return quant_rows_e4m3(L, w, rows, cols, static_cast<uint8_t*>(q), scale);
}

}  // extern "C"

// ---------------------------------------------------------------- bias gradients without allocation
// The per-slice partial sums of the bias-gradient reduction live in this fixed
// device array instead of the caller's workspace.  Host code may not pass the
// symbol itself to a kernel (on the host it is only a stand-in); the device
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) float g_bias_static[RNN_BIAS_STATIC_FLOATS];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
float* g_static_ptr[kMaxDevices] = {};

int static_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RNN_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bias_static) != cudaSuccess || !p) return RNN_ERR_CUDA;
    g_static_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_static_ptr[dev];
  return RNN_OK;
}
}  // namespace

extern "C" int rnn_bias_grad_static(rnn_handle_t h, const void* reserve, float* dw, int accumulate,
                                    cudaStream_t stream) {
  if (!h || !reserve || !dw || !aligned16(reserve) || !aligned16(dw)) return RNN_ERR_INVALID_ARG;
  const rnn_desc_t& d = h->d;
  const int GH = h->GH;
  if ((long long)GH > (long long)RNN_BIAS_STATIC_FLOATS) return RNN_ERR_UNSUPPORTED;
  if (!h->have_device) return RNN_ERR_CUDA;
  float* part = nullptr;
  RNN_TRY(static_scratch(&part));
  // every slice entry is written before it is read: nothing needs clearing
  const long long TB = (long long)d.T * d.B;
  int slices = (int)std::min<long long>(64, (TB + 255) / 256);
  slices = std::max(1, std::min(slices, RNN_BIAS_STATIC_FLOATS / GH));
  const char* R = static_cast<const char*>(reserve);
  // one bias block pair per (layer, direction) v = l * D + d, as rnn_bwd_weights writes them
  for (int v = 0; v < h->V(); ++v) {
    Launch Lb = mk(h, stream, nullptr, "bias_grad_static");
    Lb.prof = nullptr;
    RNN_TRY(bias_grad(Lb, d.mode, d.cell, d.hidden, h->u, TB, R + h->rl[v].dgx, R + h->rl[v].dgh,
                      dw + h->ul[v].bx, dw + h->ul[v].bh, accumulate, part, slices));
  }
  return RNN_OK;
}
