// Launch sequences of the backward and the forward for one (D, Dv), shared by the translation
// units of libfa_back.so: fa_back.cu (argument checks, workspace plan, entry points) and the
// fa_shapes_*.cu units, which instantiate the sequences of one head size D, plain or with the
// score extensions (so that they compile in parallel).  Host code, plus the kernels' headers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "fa_dq_raw.cuh"
#include "fa_fwd.cuh"
#include "fa_kernels.cuh"
#include "fa_lse_pair.cuh"

namespace fab {

struct Plan {
  int G, R, nQT, BK, nKT, nsplit, kt_per_split, nsplit_dq;
  int nblk_stats, nbv;
  int pre;  // 1: binary16 K'/V' copies in the workspace feed the row passes by TMA
  int dsq;  // 1 (with pre): the dK/dV pass stores dS and dQ is one product over it (k_dq_gemm)
  int ldds; // 64-key tiles per stored dS row tile (whole gradient-pass key tiles)
  int nsm;
  size_t off_stats, off_rmean, off_rsh, off_dOr, off_lamr, off_lse2, off_dlt, off_sg, off_part, off_dqpart, off_q16,
      off_do16, off_bstat, off_vsum, off_kd, off_vd, off_ds, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int block_keys(int D, int Dv) { return (D + Dv <= 256) ? 128 : 64; }

// Key tile of the LSE pass: 128 keys for every head size (its operands live in tensor memory,
// so N = 128 products fit; they run at twice the rate per flop of N = 64 products).
constexpr int kBKLse = 128;

// ------------------------------------------------------------------------------------------------
// tensor maps

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// binary16 tensor [d2][d1][d0] (d0 fastest); boxes of 64 x rows x 1 with the 128-byte swizzle
// (one box is one operand panel of `rows` 128-byte rows).
inline bool make_map(CUtensorMap* m, void* base, int d0, int d1, int d2, int rows = 128,
                     CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)d0 * d1 * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// ------------------------------------------------------------------------------------------------
// measurement hook: one CUDA event before the sequence and one after each launch

constexpr int kProfCalls = 256, kProfSlots = 17;
enum {
  KS_STATS = 0, KS_VSUM, KS_FINAL, KS_CONVERT, KS_PREDECODE, KS_ROWS_LSE, KS_MERGE, KS_ROWS_DQ, KS_DQ_REDUCE,
  KS_COLS, KS_DQ_GEMM, KS_STATS_IN, KS_FWD, KS_FWD_MERGE, KS_COLS_ROWSCALE, KS_SINK_GRAD, KS_DQ_RAW, KS_N
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  int ncalls = 0;
  cudaEvent_t ev[kProfCalls][kProfSlots + 1];
  int order[kProfCalls][kProfSlots];  // slots in launch order
  int nmarks[kProfCalls];
  bool created = false;
};
extern Profiler g_prof;  // defined in fa_back.cu

// Per-call recorder: mark(slot) after launching kernel `slot`.
struct CallRec {
  int call = -1;
  cudaStream_t s = nullptr;
  void begin(cudaStream_t st) {
    s = st;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (!g_prof.on || g_prof.ncalls >= kProfCalls) return;
    if (!g_prof.created) {
      for (int c = 0; c < kProfCalls; ++c)
        for (int k = 0; k <= kProfSlots; ++k) cudaEventCreate(&g_prof.ev[c][k]);
      g_prof.created = true;
    }
    call = g_prof.ncalls++;
    g_prof.nmarks[call] = 0;
    cudaEventRecord(g_prof.ev[call][kProfSlots], s);  // start marker
  }
  // kernel `slot` was just launched: its duration is measured from the previous marker
  void mark(int slot) {
    if (call < 0 || g_prof.nmarks[call] >= kProfSlots) return;
    cudaEventRecord(g_prof.ev[call][slot], s);
    g_prof.order[call][g_prof.nmarks[call]++] = slot;
  }
};

// Raw cache rows of one tensor as a 3D map (row elements, KV head, key), elements of 2, 4 or 8
// bytes so that one row is at most 256 elements; boxes cover one head and KE keys.
inline bool make_raw_map(CUtensorMap* m, const void* base, long rb, int Hkv, int M, int ke) {
  auto fn = encode_fn();
  if (!fn) return false;
  int es = 2;
  while (rb / es > 256) es *= 2;
  const CUtensorMapDataType dt =
      es == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : es == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_INT64;
  cuuint64_t dims[3] = {(cuuint64_t)(rb / es), (cuuint64_t)Hkv, (cuuint64_t)M};
  cuuint64_t strides[2] = {(cuuint64_t)rb, (cuuint64_t)rb * Hkv};
  cuuint32_t box[3] = {(cuuint32_t)(rb / es), 1, (cuuint32_t)ke};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// ------------------------------------------------------------------------------------------------
// launch sequence for one (D, Dv)

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Raw K/V staging of the row passes: entry size (keys) and the depths of the K and V rings
// that fit the budget.  Both rings get the same depth, and bytes left over go to extra K
// entries (the K rows of the next tile are what the decoders need first).
inline void pick_raw(Params& q, int budget, int BK) {
  const int pair = q.rbk_pad + q.rbv_pad;
  // the largest entry (fewest waits) of which two of both tensors and a third K entry fit,
  // else 32 keys
  int ke = std::min(32, BK);
  for (int c = BK; c > 32; c >>= 1)
    if (2 * c * pair + c * q.rbk_pad <= budget) {
      ke = c;
      break;
    }
  while (ke > 1 && 2 * ke * pair > budget) ke >>= 1;
  q.ke = ke;
  int d = std::max(1, std::min(kMaxRawDepth, budget / std::max(1, ke * pair)));
  q.raw_depth = q.raw_depth_v = d;
  while (q.raw_depth < kMaxRawDepth && (q.raw_depth + 1) * ke * q.rbk_pad + d * ke * q.rbv_pad <= budget)
    ++q.raw_depth;
}

inline int raw_bytes(const Params& q) { return q.ke * (q.raw_depth * q.rbk_pad + q.raw_depth_v * q.rbv_pad); }

// The LSE/D pass on CTA pairs from the raw cache (k_lse_pair), then the merge.  Needs raw rows
// that TMA can box (16-byte multiples); returns cudaErrorNotSupported otherwise, before launching.
template <int D, int Dv, bool EXT>
cudaError_t lse_pair(Params pl, const Plan& P, cudaStream_t s, CallRec& rec) {
  using L = LsePairCfg<D, Dv>;
  if (!pl.raw_bulk) return cudaErrorNotSupported;
  pick_raw(pl, L::RAW_BUDGET, L::HK);
  if (L::HK % pl.ke || (pl.ke * pl.rbk_pad) % 128 || (pl.ke * pl.rbv_pad) % 128) return cudaErrorNotSupported;
  const int sm = L::OFF_RAW + raw_bytes(pl) + 1024 + 64;  // + base alignment, decoders' realigning reads
  if (sm > 232448) return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!make_raw_map(&tk, pl.k, pl.rbk, pl.Hkv, pl.M, pl.ke) || !make_raw_map(&tv, pl.v, pl.rbv, pl.Hkv, pl.M, pl.ke))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = set_smem(k_lse_pair<D, Dv, EXT>, sm)) != cudaSuccess) return e;
  // the kernel's per-warpgroup register split must fit the registers it is launched with, or a
  // warpgroup would wait for registers that never come free
  static const int launch_regs = [] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, k_lse_pair<D, Dv, EXT>) == cudaSuccess ? fa.numRegs : 0;
  }();
  if ((long)launch_regs * L::NT < L::REG_NEED) return cudaErrorInvalidConfiguration;
  k_lse_pair<D, Dv, EXT><<<dim3(2 * ((P.nQT + 1) / 2), pl.Hkv, P.nsplit), L::NT, sm, s>>>(tk, tv, pl);
  rec.mark(KS_ROWS_LSE);
  k_lse_merge<<<(unsigned)(((long)pl.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
  rec.mark(KS_MERGE);
  return cudaGetLastError();
}

// k_predecode's grid: x walks the keys (each block step covers at least 8 keys), y = 2 * Hkv
// (the K' and V' heads); about 16 blocks per SM in all.
inline dim3 predecode_grid(const Params& p, int nsm) {
  const long gx = std::max(1L, std::min((16L * nsm) / (2L * p.Hkv), ((long)p.M + 7) / 8));
  return dim3((unsigned)gx, (unsigned)(2 * p.Hkv));
}

// Row passes over the binary16 K'/V' copies (written here by k_predecode), fed by TMA.
template <int D, int Dv, int BK, int BKL, bool EXT>
cudaError_t rows_pre(const Params& pl, const Params& pq, const Plan& P, const CUtensorMap& tmQ, dim3 grid,
                            cudaStream_t s, CallRec& rec) {
  using FL = Rows3Cfg<D, Dv, BKL, 0>;
  using FQ = Rows3Cfg<D, Dv, BK, 1>;
  CUtensorMap tkl, tvl, tkq, tvq;
  // panel-major copies: [Hkv * D/64 panels][M keys][64 columns]
  if (!make_map(&tkl, pl.kd, 64, pl.M, pl.Hkv * (D / 64), BKL) ||
      !make_map(&tvl, pl.vd, 64, pl.M, pl.Hkv * (Dv / 64), BKL) ||
      !make_map(&tkq, pq.kd, 64, pq.M, pq.Hkv * (D / 64), BK) || !make_map(&tvq, pq.vd, 64, pq.M, pq.Hkv * (Dv / 64), BK))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = set_smem(k_rows3<D, Dv, BKL, 0, EXT>, FL::SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(k_rows3<D, Dv, BK, 1, EXT>, FQ::SMEM)) != cudaSuccess) return e;
  k_predecode<<<predecode_grid(pl, P.nsm), 256, 0, s>>>(pl);
  rec.mark(KS_PREDECODE);
  if (!pl.lse_in) {  // else the per-row values come from the given lse and delta
    k_rows3<D, Dv, BKL, 0, EXT><<<grid, FL::NT, FL::SMEM, s>>>(tmQ, tkl, tvl, pl);
    rec.mark(KS_ROWS_LSE);
    k_lse_merge<<<(unsigned)(((long)pl.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
    rec.mark(KS_MERGE);
  }
  if (!P.dsq) {  // else dQ comes from the stored dS after the dK/dV pass
    k_rows3<D, Dv, BK, 1, EXT><<<grid, FQ::NT, FQ::SMEM, s>>>(tmQ, tkq, tvq, pq);
    rec.mark(KS_ROWS_DQ);
  }
  return cudaSuccess;
}

// Row passes that stage raw cache rows in shared memory and decode them there.
template <int D, int Dv, int BK, int BKL, bool EXT>
cudaError_t rows_raw(Params pl, Params pq, const Plan& P, const CUtensorMap& tmQ, dim3 grid, cudaStream_t s,
                            CallRec& rec) {
  using RL = Rows2Cfg<D, Dv, BKL, 0>;
  using RQ = Rows2Cfg<D, Dv, BK, 1>;
  static_assert(RL::RAW_BUDGET > 0 && RQ::RAW_BUDGET > 0, "shared memory budget");
  static_assert(RL::TCOLS <= 512 && RQ::TCOLS <= 512, "tensor memory budget");
  pick_raw(pl, RL::RAW_BUDGET, BKL);
  pick_raw(pq, RQ::RAW_BUDGET, BK);
  for (Params* q : {&pl, &pq})  // TMA destinations must start on 128-byte boundaries
    if ((q->ke * q->rbk_pad) % 128 || (q->ke * q->rbv_pad) % 128) q->raw_bulk = 0;
  // + 1024 for aligning the base, + 64 for the decoders' realigning reads past the last raw row
  const int sm_l = RL::OFF_RAW + raw_bytes(pl) + 1024 + 64;
  const int sm_q = RQ::OFF_RAW + raw_bytes(pq) + 1024 + 64;
  if (sm_l > 232448 || sm_q > 232448) return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = set_smem(k_rows2<D, Dv, BKL, 0, EXT>, sm_l)) != cudaSuccess) return e;
  if ((e = set_smem(k_rows2<D, Dv, BK, 1, EXT>, sm_q)) != cudaSuccess) return e;
  CUtensorMap tkl, tvl, tkq, tvq;
  std::memset(&tkl, 0, sizeof(tkl));
  tvl = tkq = tvq = tkl;
  if (pl.raw_bulk) {
    if (!make_raw_map(&tkl, pl.k, pl.rbk, pl.Hkv, pl.M, pl.ke) ||
        !make_raw_map(&tvl, pl.v, pl.rbv, pl.Hkv, pl.M, pl.ke) ||
        !make_raw_map(&tkq, pq.k, pq.rbk, pq.Hkv, pq.M, pq.ke) || !make_raw_map(&tvq, pq.v, pq.rbv, pq.Hkv, pq.M, pq.ke))
      return cudaErrorInvalidValue;
  }
  if (!pl.lse_in) {
    cudaError_t ep = lse_pair<D, Dv, EXT>(pl, P, s, rec);
    if (ep == cudaErrorNotSupported) {
      k_rows2<D, Dv, BKL, 0, EXT><<<grid, RL::NT, sm_l, s>>>(tmQ, tkl, tvl, pl);
      rec.mark(KS_ROWS_LSE);
      k_lse_merge<<<(unsigned)(((long)pl.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
      rec.mark(KS_MERGE);
    } else if (ep != cudaSuccess) {
      return ep;
    }
  }
  if (!P.dsq) {  // else dQ comes from the stored dS after the dK/dV pass
    k_rows2<D, Dv, BK, 1, EXT><<<grid, RQ::NT, sm_q, s>>>(tmQ, tkq, tvq, pq);
    rec.mark(KS_ROWS_DQ);
  }
  return cudaSuccess;
}

// Raw K staging of k_dq_raw: the largest entry (a whole key tile, else halves down to 32 keys)
// of which at least two fit the budget, and as many entries as fit (at most kMaxRawDepth).
inline void pick_raw_k(Params& q, int budget, int BK) {
  int ke = BK;
  while (ke > 32 && 2 * ke * q.rbk_pad > budget) ke >>= 1;
  while (ke > 1 && 2 * ke * q.rbk_pad > budget) ke >>= 1;
  q.ke = ke;
  q.raw_depth = std::max(1, std::min(kMaxRawDepth, budget / std::max(1, ke * q.rbk_pad)));
}

// dQ over the stored dS with K decoded from the raw cache (k_dq_raw): two row tiles per CTA.
template <int D, int BK>
cudaError_t dq_raw(Params pr, const Plan& P, const CUtensorMap& tmS, cudaStream_t s, CallRec& rec) {
  using QC = DqRawCfg<D, BK>;
  pick_raw_k(pr, QC::RAW_BUDGET, BK);
  if ((pr.ke * pr.rbk_pad) % 128) pr.raw_bulk = 0;  // TMA destinations start on 128-byte boundaries
  if (pr.raw_depth < 2 || BK % pr.ke) return cudaErrorInvalidValue;
  CUtensorMap tk;
  std::memset(&tk, 0, sizeof(tk));
  if (pr.raw_bulk && !make_raw_map(&tk, pr.k, pr.rbk, pr.Hkv, pr.M, pr.ke)) return cudaErrorInvalidValue;
  // + 1024 for aligning the base, + 64 for the decoders' realigning reads past the last raw row
  const int sm = QC::OFF_RAW + pr.ke * pr.raw_depth * pr.rbk_pad + 1024 + 64;
  if (sm > QC::SMEM_MAX) return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = set_smem(k_dq_raw<D, BK>, sm)) != cudaSuccess) return e;
  k_dq_raw<D, BK><<<dim3((P.nQT + 1) / 2, pr.Hkv, pr.nsplit), QC::NT, sm, s>>>(tmS, tk, pr);
  rec.mark(KS_DQ_RAW);
  return cudaSuccess;
}

template <int D, int Dv, bool EXT>
cudaError_t run_shape(const Params& p, const Plan& P, const CUtensorMap& tmQ, const CUtensorMap& tmO,
                             cudaStream_t s, CallRec& rec) {
  constexpr int BK = (D + Dv <= 256) ? 128 : 64;
  constexpr int BKL = kBKLse;  // LSE-pass key tile
  static_assert(BKL % BK == 0, "LSE tiles cover whole gradient-pass tiles");
  using CC = Cols2Cfg<D, Dv, BK>;
  static_assert(CC::SMEM <= 232448 && CC::TCOLS <= 512, "dK/dV pass budgets");
  Params pl = p, pq = p;
  // the LSE pass walks the same key splits in BKL-key tiles (split sizes are multiples of BKL)
  pl.nKT = (p.M + BKL - 1) / BKL;
  pl.kt_per_split = p.kt_per_split / (BKL / BK);
  const dim3 grid(P.nQT, p.Hkv, P.nsplit);
  cudaError_t e = P.pre ? rows_pre<D, Dv, BK, BKL, EXT>(pl, pq, P, tmQ, grid, s, rec)
                        : rows_raw<D, Dv, BK, BKL, EXT>(pl, pq, P, tmQ, grid, s, rec);
  if (e != cudaSuccess) return e;
  if (p.dsinks) {  // the sink-logit gradient from the merge's per-row terms
    k_sink_grad<<<p.H, 256, 0, s>>>(p);
    rec.mark(KS_SINK_GRAD);
  }
  // stored dS (level 2 only): contiguous 128-row x 64-key tiles, tile (hk, row tile, key tile)
  // at index (hk * nQT + qt) * ldds + kt64; one TMA box is one tile
  CUtensorMap tmS;
  std::memset(&tmS, 0, sizeof(tmS));
  if (P.dsq && !make_map(&tmS, p.ds, 64, 128, p.Hkv * P.nQT * p.ldds)) return cudaErrorInvalidValue;
  // the binary16 K'/V' copies as key tiles of the dK/dV pass (levels 2 and 1)
  CUtensorMap tkc, tvc;
  std::memset(&tkc, 0, sizeof(tkc));
  tvc = tkc;
  if (P.pre && (!make_map(&tkc, p.kd, 64, p.M, p.Hkv * (D / 64), BK) ||
                !make_map(&tvc, p.vd, 64, p.M, p.Hkv * (Dv / 64), BK)))
    return cudaErrorInvalidValue;
  if (P.nKT > 0) {
    if ((e = set_smem(k_cols2<D, Dv, BK, false, EXT>, CC::SMEM)) != cudaSuccess) return e;
    k_cols2<D, Dv, BK, false, EXT><<<dim3(P.nKT, p.Hkv), 384, CC::SMEM, s>>>(tmQ, tmO, tmS, tkc, tvc, p);
    rec.mark(KS_COLS);
    if (P.dsq) {  // the variant with per-row multipliers on the stored dS (returns at once if not needed)
      if ((e = set_smem(k_cols2<D, Dv, BK, true, EXT>, CC::SMEM)) != cudaSuccess) return e;
      k_cols2<D, Dv, BK, true, EXT><<<dim3(P.nKT, p.Hkv), 384, CC::SMEM, s>>>(tmQ, tmO, tmS, tkc, tvc, p);
      rec.mark(KS_COLS_ROWSCALE);
    }
  }
  if (P.dsq && P.pre) {
    using GC = GemmCfg<D, BK>;
    CUtensorMap tkg;
    if (!make_map(&tkg, p.kd, 64, p.M, p.Hkv * (D / 64), BK)) return cudaErrorInvalidValue;
    if ((e = set_smem(k_dq_gemm<D, BK>, GC::SMEM)) != cudaSuccess) return e;
    k_dq_gemm<D, BK><<<grid, 256, GC::SMEM, s>>>(tmS, tkg, p);
    rec.mark(KS_DQ_GEMM);
  } else if (P.dsq) {  // no K' copy: the dQ product decodes raw K tiles itself
    // with key splits of its own: its grid has half as many row units, so the plan's split count
    // can leave a mostly empty last wave; the count that fills whole waves best (at most the
    // plan's, whose partial buffer it writes), by the plan's cost of waves per split
    Params pr = p;
    const long units = (long)((P.nQT + 1) / 2) * p.Hkv;
    int ns = P.nsplit;
    double best = 1e30;
    for (int c = 1; c <= P.nsplit; ++c) {
      const double cost = (double)((units * c + P.nsm - 1) / P.nsm) / c * (1.0 + 0.01 * c);
      if (cost < best - 1e-12) best = cost, ns = c;
    }
    pr.kt_per_split = (P.nKT + ns - 1) / ns;
    pr.nsplit = P.nKT > 0 ? (P.nKT + pr.kt_per_split - 1) / pr.kt_per_split : 1;
    if ((e = dq_raw<D, BK>(pr, P, tmS, s, rec)) != cudaSuccess) return e;
    if (pr.nsplit > 1) {
      k_dq_reduce<<<(unsigned)(((long)p.Hkv * P.R * (D / 4) + 255) / 256), 256, 0, s>>>(pr);
      rec.mark(KS_DQ_REDUCE);
    }
    return cudaGetLastError();
  }
  if (P.nsplit_dq > 1) {
    k_dq_reduce<<<(unsigned)(((long)p.Hkv * P.R * (D / 4) + 255) / 256), 256, 0, s>>>(p);
    rec.mark(KS_DQ_REDUCE);
  }
  return cudaGetLastError();
}

// Forward: the one-pass kernel (online softmax, O accumulated in tensor memory) over the binary16
// K'/V' copies in 64-key tiles, then, with key splits, the fixed-order merge of the partials.
// Plan level 1 (the copies, no stored dS).
template <int D, int Dv>
cudaError_t run_forward(const Params& p, const Plan& P, const CUtensorMap&, const CUtensorMap&,
                        cudaStream_t s, CallRec& rec) {
  using F = Fwd1Cfg<D, Dv>;
  Params pf = p;
  pf.nKT = (p.M + F::BK - 1) / F::BK;
  pf.kt_per_split = p.kt_per_split * (P.BK / F::BK);  // the plan's splits in 64-key tiles
  CUtensorMap tk, tv;
  if (!make_map(&tk, p.kd, 64, p.M, p.Hkv * (D / 64), F::BK) || !make_map(&tv, p.vd, 64, p.M, p.Hkv * (Dv / 64), F::BK))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = set_smem(k_fwd1<D, Dv>, F::SMEM)) != cudaSuccess) return e;
  k_predecode<<<predecode_grid(p, P.nsm), 256, 0, s>>>(p);
  rec.mark(KS_PREDECODE);
  k_fwd1<D, Dv><<<dim3(P.nQT, p.Hkv, P.nsplit), F::NT, F::SMEM, s>>>(tk, tv, pf);
  rec.mark(KS_FWD);
  if (P.nsplit > 1) {
    k_fwd_merge<<<(unsigned)(((long)p.Hkv * P.R * (Dv / 4) + 255) / 256), 256, 0, s>>>(pf);
    rec.mark(KS_FWD_MERGE);
  }
  return cudaGetLastError();
}

using RunFn = cudaError_t (*)(const Params&, const Plan&, const CUtensorMap&, const CUtensorMap&, cudaStream_t,
                              CallRec&);

// The sequence of head sizes (D, Dv): the forward or the plain backward (pick_plain), or the
// backward with the score extensions (pick_ext: the EXT variants of the score-forming kernels).
// Null for an unsupported Dv.
template <int D>
RunFn pick_plain(int Dv, bool forward) {
  switch (Dv) {
    case 64: return forward ? run_forward<D, 64> : run_shape<D, 64, false>;
    case 128: return forward ? run_forward<D, 128> : run_shape<D, 128, false>;
    case 256: return forward ? run_forward<D, 256> : run_shape<D, 256, false>;
  }
  return nullptr;
}
template <int D>
RunFn pick_ext(int Dv) {
  switch (Dv) {
    case 64: return run_shape<D, 64, true>;
    case 128: return run_shape<D, 128, true>;
    case 256: return run_shape<D, 256, true>;
  }
  return nullptr;
}
// one translation unit each (fa_shapes_d<D>.cu, fa_shapes_d<D>_ext.cu)
RunFn pick_d64(int Dv, bool forward);
RunFn pick_d128(int Dv, bool forward);
RunFn pick_d256(int Dv, bool forward);
RunFn pick_d64_ext(int Dv);
RunFn pick_d128_ext(int Dv);
RunFn pick_d256_ext(int Dv);

}  // namespace fab
