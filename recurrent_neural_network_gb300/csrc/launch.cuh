// launch.cuh -- host templates that turn an (Operand, Operand, epilogue) triple
// into a launch of one of the two GEMM engines.  Included by the kernel
// translation units only.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "../../include/rnn.h"
#include "engine.cuh"
#include "launchers.h"

namespace rnn {

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime.
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D bf16 tensor map over an operand with 128-byte swizzle.  K-major operands
// use a box of 64 (k) x box_rows (mn); MN-major operands a box of 64 (mn) x 64 (k).
// An MN-major operand whose MN extent is a multiple of 64 gets a 3-D map
// (64 MN, K, MN / 64) with box (64, 64, box_rows / 64), *three_d = 1: one
// load brings all 64-wide blocks of a tile, in the same shared-memory image
// (block j at j x 8 KB, 128-byte swizzle) the per-block 2-D loads write (a
// TMA load costs about the same to issue whatever its size).
inline int encode_operand(CUtensorMap* map, const Operand& op, int box_rows, int* three_d = nullptr) {
  auto enc = tmap_encoder();
  if (!enc) return RNN_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(op.ptr) & 15) || ((op.ld * 2) & 15)) return RNN_ERR_INVALID_ARG;
  if (three_d) *three_d = 0;
  if (three_d && op.mn_major && box_rows > 64 && box_rows % 64 == 0 && op.mn_ext % 64 == 0) {
    cuuint64_t dims3[3] = {64, (cuuint64_t)op.k_ext, (cuuint64_t)(op.mn_ext / 64)};
    cuuint64_t strides3[2] = {(cuuint64_t)op.ld * 2, 128};
    cuuint32_t box3[3] = {64, 64, (cuuint32_t)(box_rows / 64)}, es3[3] = {1, 1, 1};
    const CUresult r3 = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims3, strides3, box3,
                            es3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r3 == CUDA_SUCCESS) {
      *three_d = 1;
      return RNN_OK;
    }
  }
  cuuint64_t dims[2], strides[1];
  cuuint32_t box[2], es[2] = {1, 1};
  if (op.mn_major) {
    dims[0] = (cuuint64_t)op.mn_ext;
    dims[1] = (cuuint64_t)op.k_ext;
    box[0] = 64;
    box[1] = 64;
  } else {
    dims[0] = (cuuint64_t)op.k_ext;
    dims[1] = (cuuint64_t)op.mn_ext;
    box[0] = 64;
    box[1] = (cuuint32_t)box_rows;
  }
  strides[0] = (cuuint64_t)op.ld * 2;
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(op.ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RNN_OK : RNN_ERR_INVALID_ARG;
}

// 2-D tensor map without swizzle over a row-major rows x cols array of
// fp32 (elem 4) or bf16 (elem 2) with row pitch ld elements; box box_cols x
// box_rows.  Used for the bulk stores and loads of epilogues.
inline int encode_plain(CUtensorMap* map, const void* ptr, int elem, long long rows, long long cols, long long ld,
                        int box_cols, int box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return RNN_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || ((ld * elem) & 15) || ((box_cols * elem) & 15))
    return RNN_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows}, strides[1] = {(cuuint64_t)(ld * elem)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows}, es[2] = {1, 1};
  CUresult r = enc(map, elem == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RNN_OK : RNN_ERR_INVALID_ARG;
}

inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RNN_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorLaunchOutOfResources) return RNN_ERR_LAUNCH;
  return RNN_ERR_CUDA;
}

// Launch attributes of a tcgen05 engine launch: a cluster shape when the
// cluster has more than one CTA, and programmatic stream serialization when
// the kernel may start while the previous kernel on the stream is finishing
// (the engine waits on the grid dependency before it touches produced data).
inline unsigned launch_attrs(cudaLaunchAttribute* at, int cluster, int pdl) {
  unsigned n = 0;
  if (cluster > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  return n;
}

// cluster_splitk: with more than one K split, the splits of each output tile
// run as one thread-block cluster and reduce through distributed shared
// memory (the epilogue must support it); one tile per CTA.
template <int BN, int STAGES, class Epi>
int launch_tc(const Launch& L, const Operand& A, const Operand& B, int M, int N, int K, int splits, int max_ctas,
              const Epi& epi, bool cluster_splitk = false) {
  if (M <= 0 || N <= 0 || K <= 0) return RNN_ERR_INVALID_ARG;
  if (B.mn_major && BN % 64) return RNN_ERR_UNSUPPORTED;
  CUtensorMap ma, mb;
  int a3 = 0, b3 = 0;
  int rc = encode_operand(&ma, A, tce::BM, &a3);
  if (rc) return rc;
  rc = encode_operand(&mb, B, BN, &b3);
  if (rc) return rc;
  GemmGeom g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + tce::BM - 1) / tce::BM;
  g.n_tiles = (N + BN - 1) / BN;
  g.kb_total = (K + tce::BK - 1) / tce::BK;
  splits = std::max(1, std::min(splits, g.kb_total));
  g.kb_per_split = (g.kb_total + splits - 1) / splits;
  g.splits = (g.kb_total + g.kb_per_split - 1) / g.kb_per_split;
  g.num_tiles = g.m_tiles * g.n_tiles * g.splits;
  g.a_mn = A.mn_major;
  g.b_mn = B.mn_major;
  g.a3 = a3;
  g.b3 = b3;
  g.limit_ns = L.limit_ns;
  g.err = L.err;
  g.steps = 1;
  g.tiles_per_step = 0;
  g.b_step_rows = 0;
  g.step_cnt = nullptr;
  g.step_want = 0;
  // The cluster reduction gives each CTA BN/splits columns, read as 16-byte
  // vectors and processed 16 hidden units at a time: it needs BN to be a
  // multiple of 16*splits and at most 8 CTAs per cluster.  Otherwise the
  // partials go through global memory.
  g.cluster = (cluster_splitk && g.splits > 1 && g.splits <= 8 && BN % (16 * g.splits) == 0) ? g.splits : 1;
  // tile order: run along the dimension with fewer tiles first, so that the
  // CTAs in flight at any time share operand slabs of the other dimension
  // (for the deep-K products this keeps the slabs they stream in L2)
  g.nfast = g.n_tiles < g.m_tiles ? 1 : 0;
  constexpr int smem = tce::smem_bytes<BN, STAGES>();
  auto kern = tc_gemm_kernel<BN, STAGES, Epi>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_status(e);
    attr = true;
  }
  int cap = max_ctas > 0 ? max_ctas : L.num_sms;
  const int grid = std::min(g.num_tiles, cap);
  g.pdl = L.pdl;
  g.static_op = A.is_static ? 1 : B.is_static ? 2 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.cluster > 1 ? g.num_tiles : grid);
  cfg.blockDim = dim3(64 + 32 * EpiWarps<Epi>::value);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute at[2];
  cfg.attrs = at;
  cfg.numAttrs = launch_attrs(at, g.cluster, L.pdl);
  launch_begin(L);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, g, epi);
  launch_end(L);
  return cuda_status(e);
}

// CTA-pair engine: 256 x BN tiles over clusters of 2 CTAs.  With splits > 1
// the K splits of a tile run as one cluster of 2*splits CTAs (pairs at ranks
// 2i, 2i+1) and reduce through distributed shared memory (the epilogue must
// support it); RNN_ERR_UNSUPPORTED when the split cannot be laid out so.
// steps > 1: the products of `steps` dependent steps in one cooperative
// launch, one tile per pair and step (see GemmGeom::steps); B's rows of step
// s at b_step_rows * s; the epilogue of each tile arrives tile_arrivals times
// on step_cnt[s]; RNN_ERR_UNSUPPORTED where a step's tiles outnumber the pairs.
template <int BN, int STAGES, class Epi, int ACCS = 2>
int launch_tc2(const Launch& L, const Operand& A, const Operand& B, int M, int N, int K, int max_ctas,
               const Epi& epi, int splits = 1, int steps = 1, int b_step_rows = 0, unsigned int* step_cnt = nullptr,
               unsigned int tile_arrivals = 0) {
  if (M <= 0 || N <= 0 || K <= 0) return RNN_ERR_INVALID_ARG;
  if (B.mn_major && (BN / 2) % 64) return RNN_ERR_UNSUPPORTED;
  CUtensorMap ma, mb;
  int a3 = 0, b3 = 0;
  int rc = encode_operand(&ma, A, 128, &a3);
  if (rc) return rc;
  rc = encode_operand(&mb, B, BN / 2, &b3);
  if (rc) return rc;
  GemmGeom g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + tce2::BM - 1) / tce2::BM;
  g.n_tiles = (N + BN - 1) / BN;
  g.kb_total = (K + tce2::BK - 1) / tce2::BK;
  splits = std::max(1, std::min(splits, g.kb_total));
  g.kb_per_split = (g.kb_total + splits - 1) / splits;
  g.splits = (g.kb_total + g.kb_per_split - 1) / g.kb_per_split;
  if (g.splits > 1 && (g.splits > 4 || BN % (16 * g.splits))) return RNN_ERR_UNSUPPORTED;
  g.num_tiles = g.m_tiles * g.n_tiles * g.splits;
  g.a_mn = A.mn_major;
  g.b_mn = B.mn_major;
  g.a3 = a3;
  g.b3 = b3;
  g.limit_ns = L.limit_ns;
  g.err = L.err;
  g.steps = 1;
  g.tiles_per_step = 0;
  g.b_step_rows = 0;
  g.step_cnt = nullptr;
  g.step_want = 0;
  g.cluster = g.splits;
  g.nfast = g.n_tiles < g.m_tiles ? 1 : 0;  // as in launch_tc
  constexpr int smem = tce2::smem_bytes<BN, STAGES>();
  auto kern = tc_gemm2_kernel<BN, STAGES, Epi, ACCS>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_status(e);
    attr = true;
  }
  const int cap = (max_ctas > 0 ? max_ctas : L.num_sms) / 2;
  // split-K: one tile per pair so that the cluster reduction can reuse the stages
  int pairs = g.cluster > 1 ? g.num_tiles : std::max(1, std::min(g.num_tiles, cap));
  if (steps > 1) {
    if (g.cluster > 1 || g.num_tiles > cap || !step_cnt) return RNN_ERR_UNSUPPORTED;
    g.steps = steps;
    g.tiles_per_step = g.num_tiles;
    g.b_step_rows = b_step_rows;
    g.step_cnt = step_cnt;
    g.step_want = tile_arrivals * static_cast<unsigned int>(g.num_tiles);
    pairs = g.num_tiles;
    g.num_tiles *= steps;
  }
  // (a cooperative launch is never a programmatic dependent)
  const int pdl = steps > 1 ? 0 : L.pdl;
  g.pdl = pdl;
  g.static_op = A.is_static ? 1 : B.is_static ? 2 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(64 + 32 * EpiWarps<Epi>::value);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute at[3];
  cfg.attrs = at;
  cfg.numAttrs = launch_attrs(at, 2 * g.cluster, pdl);
  if (steps > 1) {
    // the pairs wait on one another's stores: all of them resident at once
    at[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
    at[cfg.numAttrs].val.cooperative = 1;
    ++cfg.numAttrs;
  }
  launch_begin(L);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, g, epi);
  launch_end(L);
  return cuda_status(e);
}

template <int BN, class Epi>
int launch_simt(const Launch& L, const Operand& A, const Operand& B, int M, int N, int K, const Epi& epi) {
  if (M <= 0 || N <= 0 || K <= 0) return RNN_ERR_INVALID_ARG;
  GemmGeom g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + se::BM - 1) / se::BM;
  g.n_tiles = (N + BN - 1) / BN;
  g.splits = 1;
  g.kb_total = (K + se::BK - 1) / se::BK;
  g.kb_per_split = g.kb_total;
  g.num_tiles = g.m_tiles * g.n_tiles;
  g.cluster = 1;
  g.nfast = 0;
  g.pdl = 0;
  g.static_op = 0;
  g.a_mn = A.mn_major;
  g.b_mn = B.mn_major;
  g.a3 = 0;
  g.b3 = 0;
  g.limit_ns = L.limit_ns;
  g.err = L.err;
  g.steps = 1;
  g.tiles_per_step = 0;
  g.b_step_rows = 0;
  g.step_cnt = nullptr;
  g.step_want = 0;
  constexpr int smem = se::smem_bytes<BN>();
  auto kern = simt_gemm_kernel<BN, Epi>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_status(e);
    attr = true;
  }
  launch_begin(L);
  kern<<<g.num_tiles, 128, smem, L.stream>>>(static_cast<const float*>(A.ptr), A.ld,
                                             static_cast<const float*>(B.ptr), B.ld, g, epi);
  cudaError_t e = cudaGetLastError();
  launch_end(L);
  return cuda_status(e);
}

}  // namespace rnn
