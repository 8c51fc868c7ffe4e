// Host side of the flash-attention backward: argument checks, workspace layout, TMA tensor
// maps and the launch sequence behind the C ABI declared in include/fa_back.h.
//
// Numerics (the reading of "CUDA: FLASH_ATTN_BACK kernels", CambrianTech/llama.cpp pull
// request 63, for a binary16 tensor-core path):
//  * every contraction runs as binary16 x binary16 -> f32 on tcgen05 (kind::f16);
//  * Q, dO, K^, V^ are multiplied by powers of two (max magnitude below 2^14) before rounding,
//    P by 2^15 and dS by a power of two derived from a norm bound, so no operand leaves the
//    binary16 normal range and the scales divide out exactly;
//  * V^ is shifted by its column mean r per KV head: dP'_ij = dO_i . (v^_j - r).  Since the
//    softmax weights of a row sum to one, dP'_ij - delta'_i = dP_ij - delta_i, and the reported
//    delta adds dO_i . r back.  The rounded operand then carries V's variation at binary16's
//    relative precision, which the near-constant-V case needs;
//  * dS = p * (dP' - delta') is formed by direct f32 subtraction (review of revision a0ea747);
//  * the softmax statistics (running max, sum, sum of p*dP) use f32 with compensated chunk
//    accumulation; split partials merge in a fixed order, so results are deterministic.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <limits>
#include <mutex>

#include "../../include/fa_back.h"
#include "fa_internal.h"
#include "fa_kernels.cuh"
#include "fa_lse_pair.cuh"

namespace fab {

__device__ int g_err = 0;

struct Plan {
  int G, R, nQT, BK, nKT, nsplit, kt_per_split, nsplit_dq;
  int nblk_stats, nbv;
  int pre;  // 1: binary16 K'/V' copies in the workspace feed the row passes by TMA
  int dsq;  // 1 (with pre): the dK/dV pass stores dS and dQ is one product over it (k_dq_gemm)
  int ldds; // 64-key tiles per stored dS row tile (whole gradient-pass key tiles)
  int nsm;
  size_t off_stats, off_rmean, off_rsh, off_dOr, off_lamr, off_lse2, off_dlt, off_part, off_dqpart, off_q16, off_do16,
      off_bstat, off_vsum, off_kd, off_vd, off_ds, total;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int block_keys(int D, int Dv) { return (D + Dv <= 256) ? 128 : 64; }

// Key tile of the LSE pass: 128 keys for every head size (its operands live in tensor memory,
// so N = 128 products fit; they run at twice the rate per flop of N = 64 products).
constexpr int kBKLse = 128;

// Workspace offsets of a plan whose split counts are set.
static void layout(Plan& P, int M, int Hkv, int D, int Dv) {
  size_t o = 0;
  P.off_stats = o; o = align256(o + sizeof(Stats));
  P.off_rmean = o; o = align256(o + sizeof(float) * (size_t)Hkv * Dv);
  P.off_rsh = o; o = align256(o + sizeof(float) * (size_t)Hkv * Dv);
  P.off_dOr = o; o = align256(o + sizeof(float) * (size_t)Hkv * P.R);
  P.off_lamr = o; o = align256(o + sizeof(float) * (size_t)Hkv * P.R);
  P.off_lse2 = o; o = align256(o + sizeof(float) * (size_t)Hkv * P.R);
  P.off_dlt = o; o = align256(o + sizeof(float) * (size_t)Hkv * P.R);
  P.off_part = o; o = align256(o + sizeof(float) * 3 * (size_t)P.nsplit * Hkv * P.R);
  // split partials of dQ (backward) or O (forward)
  P.off_dqpart = o;
  o = align256(o + (P.nsplit_dq > 1 ? sizeof(float) * (size_t)P.nsplit_dq * Hkv * P.R * (D > Dv ? D : Dv) : 0));
  P.off_q16 = o; o = align256(o + 2 * (size_t)Hkv * P.R * D);
  P.off_do16 = o; o = align256(o + 2 * (size_t)Hkv * P.R * Dv);
  P.off_bstat = o; o = align256(o + sizeof(float) * 8 * (size_t)P.nblk_stats);
  P.off_vsum = o; o = align256(o + sizeof(float) * (size_t)P.nbv * Hkv * Dv);
  P.off_kd = o; o = align256(o + (P.pre ? 2 * (size_t)Hkv * M * D : 0));
  P.off_vd = o; o = align256(o + (P.pre ? 2 * (size_t)Hkv * M * Dv : 0));
  P.off_ds = o; o = align256(o + (P.dsq ? (size_t)Hkv * P.nQT * P.ldds * (128 * 64 * 2) : 0));
  P.total = o;
}

// Launch plan and workspace layout for one variant (level 2: stored dS and a dQ product over it;
// 1: binary16 K'/V' copies feeding the row passes; 0: row passes decoding the raw cache).  The
// keys of each row tile are split so that the last wave of CTAs (one per SM) wastes least,
// counting a small cost per split for the partial merges; among split counts whose workspace
// fits `ws_cap`, the cheapest is taken (1 if none fits).
static Plan plan_variant(int N, int M, int H, int Hkv, int D, int Dv, int nsm, size_t ws_cap, int level) {
  Plan P;
  std::memset(&P, 0, sizeof(P));
  P.pre = level >= 1;
  P.dsq = level >= 2;
  P.ldds = (M + block_keys(D, Dv) - 1) / block_keys(D, Dv) * (block_keys(D, Dv) / 64);  // whole key tiles
  P.nsm = nsm;
  P.G = H / Hkv;
  P.R = N * P.G;
  P.nQT = (P.R + 127) / 128;
  P.BK = block_keys(D, Dv);
  P.nKT = (M + P.BK - 1) / P.BK;
  const long rows = 2L * N * H + 2L * M * Hkv;
  P.nblk_stats = (int)std::max(1L, std::min(8L * nsm, (rows + 7) / 8));
  P.nbv = std::max(1, std::min(256, (M + 255) / 256));
  auto set_split = [&](int ns) {
    P.kt_per_split = P.nKT > 0 ? (P.nKT + ns - 1) / ns : 1;
    const int r = kBKLse / P.BK;  // whole LSE-pass tiles per split
    P.kt_per_split = (P.kt_per_split + r - 1) / r * r;
    P.nsplit = P.nKT > 0 ? (P.nKT + P.kt_per_split - 1) / P.kt_per_split : 1;
    P.nsplit_dq = P.nsplit;
    layout(P, M, Hkv, D, Dv);
  };
  const int base = std::max(1, P.nQT * Hkv);
  int ns = 1;
  double best = 1e30;
  for (int c = 1; c <= std::min(64, std::max(1, P.nKT)); ++c) {
    const double waves = (double)(((long)base * c + nsm - 1) / nsm);
    const double cost = waves / c * (1.0 + 0.01 * c);
    if (cost < best - 1e-12) {
      set_split(c);
      if (c == 1 || P.total <= ws_cap) best = cost, ns = c;
    }
  }
  set_split(ns);
  return P;
}

// The fastest plan whose workspace fits ws_cap, trying the levels from 2 down; level 0 with one
// split is the smallest workspace fa_back() accepts.
static Plan make_plan(int N, int M, int H, int Hkv, int D, int Dv, int nsm, size_t ws_cap = SIZE_MAX) {
  for (int level = 2; level > 0; --level) {
    const Plan P = plan_variant(N, M, H, Hkv, D, Dv, nsm, ws_cap, level);
    if (P.total <= ws_cap) return P;
  }
  return plan_variant(N, M, H, Hkv, D, Dv, nsm, ws_cap, 0);
}

static int device_sms(int* major, int* minor) {
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (major) cudaDeviceGetAttribute(major, cudaDevAttrComputeCapabilityMajor, dev);
  if (minor) cudaDeviceGetAttribute(minor, cudaDevAttrComputeCapabilityMinor, dev);
  return nsm;
}

// ------------------------------------------------------------------------------------------------
// tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
static bool make_map(CUtensorMap* m, void* base, int d0, int d1, int d2, int rows = 128,
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

constexpr int kProfCalls = 256, kProfSlots = 16;
// (the read-out measures each kernel from the marker recorded before it)
static const char* const kKernelNames[kProfSlots] = {
    "k_row_stats", "k_vsum", "k_finalize", "k_convert", "k_predecode", "k_rows_lse", "k_lse_merge", "k_rows_dq",
    "k_dq_reduce", "k_cols", "k_dq_gemm", "k_stats_in", "k_fwd_lse", "k_fwd_o", "k_o_reduce", "k_cols_rowscale"};
enum {
  KS_STATS = 0, KS_VSUM, KS_FINAL, KS_CONVERT, KS_PREDECODE, KS_ROWS_LSE, KS_MERGE, KS_ROWS_DQ, KS_DQ_REDUCE,
  KS_COLS, KS_DQ_GEMM, KS_STATS_IN, KS_FWD_LSE, KS_FWD_O, KS_O_REDUCE, KS_COLS_ROWSCALE, KS_N
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
static Profiler g_prof;

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
static bool make_raw_map(CUtensorMap* m, const void* base, long rb, int Hkv, int M, int ke) {
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
static cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Raw K/V staging of the row passes: entry size (keys) and the depths of the K and V rings
// that fit the budget.  Both rings get the same depth, and bytes left over go to extra K
// entries (the K rows of the next tile are what the decoders need first).
static void pick_raw(Params& q, int budget, int BK) {
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

static int raw_bytes(const Params& q) { return q.ke * (q.raw_depth * q.rbk_pad + q.raw_depth_v * q.rbv_pad); }

// The LSE/D pass on CTA pairs from the raw cache (k_lse_pair), then the merge.  Needs raw rows
// that TMA can box (16-byte multiples); returns cudaErrorNotSupported otherwise, before launching.
template <int D, int Dv>
static cudaError_t lse_pair(Params pl, const Plan& P, cudaStream_t s, CallRec& rec) {
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
  if ((e = set_smem(k_lse_pair<D, Dv>, sm)) != cudaSuccess) return e;
  k_lse_pair<D, Dv><<<dim3(2 * ((P.nQT + 1) / 2), pl.Hkv, P.nsplit), L::NT, sm, s>>>(tk, tv, pl);
  rec.mark(KS_ROWS_LSE);
  k_lse_merge<<<(unsigned)(((long)pl.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
  rec.mark(KS_MERGE);
  return cudaGetLastError();
}

// Row passes over the binary16 K'/V' copies (written here by k_predecode), fed by TMA.
template <int D, int Dv, int BK, int BKL>
static cudaError_t rows_pre(const Params& pl, const Params& pq, const Plan& P, const CUtensorMap& tmQ, dim3 grid,
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
  if ((e = set_smem(k_rows3<D, Dv, BKL, 0>, FL::SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(k_rows3<D, Dv, BK, 1>, FQ::SMEM)) != cudaSuccess) return e;
  const long units = (long)pl.M * pl.Hkv * ((D + Dv) / 8);
  k_predecode<<<(unsigned)std::min<long>((units + 255) / 256, 16L * P.nsm), 256, 0, s>>>(pl);
  rec.mark(KS_PREDECODE);
  if (!pl.lse_in) {  // else the per-row values come from the given lse and delta
    k_rows3<D, Dv, BKL, 0><<<grid, FL::NT, FL::SMEM, s>>>(tmQ, tkl, tvl, pl);
    rec.mark(KS_ROWS_LSE);
    k_lse_merge<<<(unsigned)(((long)pl.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
    rec.mark(KS_MERGE);
  }
  if (!P.dsq) {  // else dQ comes from the stored dS after the dK/dV pass
    k_rows3<D, Dv, BK, 1><<<grid, FQ::NT, FQ::SMEM, s>>>(tmQ, tkq, tvq, pq);
    rec.mark(KS_ROWS_DQ);
  }
  return cudaSuccess;
}

// Row passes that stage raw cache rows in shared memory and decode them there.
template <int D, int Dv, int BK, int BKL>
static cudaError_t rows_raw(Params pl, Params pq, const Plan& P, const CUtensorMap& tmQ, dim3 grid, cudaStream_t s,
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
  if ((e = set_smem(k_rows2<D, Dv, BKL, 0>, sm_l)) != cudaSuccess) return e;
  if ((e = set_smem(k_rows2<D, Dv, BK, 1>, sm_q)) != cudaSuccess) return e;
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
    cudaError_t ep = lse_pair<D, Dv>(pl, P, s, rec);
    if (ep == cudaErrorNotSupported) {
      k_rows2<D, Dv, BKL, 0><<<grid, RL::NT, sm_l, s>>>(tmQ, tkl, tvl, pl);
      rec.mark(KS_ROWS_LSE);
      k_lse_merge<<<(unsigned)(((long)pl.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
      rec.mark(KS_MERGE);
    } else if (ep != cudaSuccess) {
      return ep;
    }
  }
  k_rows2<D, Dv, BK, 1><<<grid, RQ::NT, sm_q, s>>>(tmQ, tkq, tvq, pq);
  rec.mark(KS_ROWS_DQ);
  return cudaSuccess;
}

template <int D, int Dv>
static cudaError_t run_shape(const Params& p, const Plan& P, const CUtensorMap& tmQ, const CUtensorMap& tmO,
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
  cudaError_t e = P.pre ? rows_pre<D, Dv, BK, BKL>(pl, pq, P, tmQ, grid, s, rec)
                        : rows_raw<D, Dv, BK, BKL>(pl, pq, P, tmQ, grid, s, rec);
  if (e != cudaSuccess) return e;
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
    if ((e = set_smem(k_cols2<D, Dv, BK, false>, CC::SMEM)) != cudaSuccess) return e;
    k_cols2<D, Dv, BK, false><<<dim3(P.nKT, p.Hkv), 384, CC::SMEM, s>>>(tmQ, tmO, tmS, tkc, tvc, p);
    rec.mark(KS_COLS);
    if (P.dsq) {  // the variant with per-row multipliers on the stored dS (returns at once if not needed)
      if ((e = set_smem(k_cols2<D, Dv, BK, true>, CC::SMEM)) != cudaSuccess) return e;
      k_cols2<D, Dv, BK, true><<<dim3(P.nKT, p.Hkv), 384, CC::SMEM, s>>>(tmQ, tmO, tmS, tkc, tvc, p);
      rec.mark(KS_COLS_ROWSCALE);
    }
  }
  if (P.dsq) {
    using GC = GemmCfg<D, BK>;
    CUtensorMap tkg;
    if (!make_map(&tkg, p.kd, 64, p.M, p.Hkv * (D / 64), BK)) return cudaErrorInvalidValue;
    if ((e = set_smem(k_dq_gemm<D, BK>, GC::SMEM)) != cudaSuccess) return e;
    k_dq_gemm<D, BK><<<grid, 256, GC::SMEM, s>>>(tmS, tkg, p);
    rec.mark(KS_DQ_GEMM);
  }
  if (P.nsplit_dq > 1) {
    k_dq_reduce<<<(unsigned)(((long)p.Hkv * P.R * (D / 4) + 255) / 256), 256, 0, s>>>(p);
    rec.mark(KS_DQ_REDUCE);
  }
  return cudaGetLastError();
}

// Forward: lse by the LSE pass without dP (MODE 3), then O += P V' per row tile with P from that
// lse (MODE 2), and the split reduce.  Plan level 1 (binary16 K'/V' copies, no stored dS).
template <int D, int Dv>
static cudaError_t run_forward(const Params& p, const Plan& P, const CUtensorMap& tmQ, const CUtensorMap&,
                               cudaStream_t s, CallRec& rec) {
  constexpr int BK = (D + Dv <= 256) ? 128 : 64;
  constexpr int BKL = kBKLse;
  using FL = Rows3Cfg<D, Dv, BKL, 3>;
  using FO = Rows3Cfg<D, Dv, BK, 2>;
  Params pl = p;
  pl.nKT = (p.M + BKL - 1) / BKL;
  pl.kt_per_split = p.kt_per_split / (BKL / BK);
  const dim3 grid(P.nQT, p.Hkv, P.nsplit);
  CUtensorMap tkl, tko, tvo;
  if (!make_map(&tkl, p.kd, 64, p.M, p.Hkv * (D / 64), BKL) || !make_map(&tko, p.kd, 64, p.M, p.Hkv * (D / 64), BK) ||
      !make_map(&tvo, p.vd, 64, p.M, p.Hkv * (Dv / 64), BK))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = set_smem(k_rows3<D, Dv, BKL, 3>, FL::SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(k_rows3<D, Dv, BK, 2>, FO::SMEM)) != cudaSuccess) return e;
  const long units = (long)p.M * p.Hkv * ((D + Dv) / 8);
  k_predecode<<<(unsigned)std::min<long>((units + 255) / 256, 16L * P.nsm), 256, 0, s>>>(p);
  rec.mark(KS_PREDECODE);
  k_rows3<D, Dv, BKL, 3><<<grid, FL::NT, FL::SMEM, s>>>(tmQ, tkl, tkl, pl);  // no V' (its map unused)
  rec.mark(KS_FWD_LSE);
  k_lse_merge<<<(unsigned)(((long)p.Hkv * P.R + 255) / 256), 256, 0, s>>>(pl);
  rec.mark(KS_MERGE);
  k_rows3<D, Dv, BK, 2><<<grid, FO::NT, FO::SMEM, s>>>(tmQ, tko, tvo, p);
  rec.mark(KS_FWD_O);
  if (P.nsplit > 1) {
    k_o_reduce<<<(unsigned)(((long)p.Hkv * P.R * (Dv / 4) + 255) / 256), 256, 0, s>>>(p);
    rec.mark(KS_O_REDUCE);
  }
  return cudaGetLastError();
}

using RunFn = cudaError_t (*)(const Params&, const Plan&, const CUtensorMap&, const CUtensorMap&, cudaStream_t,
                              CallRec&);

static RunFn pick_fwd(int D, int Dv) {
#define FAB_CASE(a, b) \
  if (D == a && Dv == b) return run_forward<a, b>;
  FAB_CASE(64, 64)
  FAB_CASE(64, 128)
  FAB_CASE(64, 256)
  FAB_CASE(128, 64)
  FAB_CASE(128, 128)
  FAB_CASE(128, 256)
  FAB_CASE(256, 64)
  FAB_CASE(256, 128)
  FAB_CASE(256, 256)
#undef FAB_CASE
  return nullptr;
}

static RunFn pick(int D, int Dv) {
#define FAB_CASE(a, b) \
  if (D == a && Dv == b) return run_shape<a, b>;
  FAB_CASE(64, 64)
  FAB_CASE(64, 128)
  FAB_CASE(64, 256)
  FAB_CASE(128, 64)
  FAB_CASE(128, 128)
  FAB_CASE(128, 256)
  FAB_CASE(256, 64)
  FAB_CASE(256, 128)
  FAB_CASE(256, 256)
#undef FAB_CASE
  return nullptr;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace fab

using namespace fab;

extern "C" long fa_row_bytes(int type, int D) {
  if (D <= 0) return -1;
  switch (type) {
    case FA_F32: return 4L * D;
    case FA_F16: return 2L * D;
    case FA_Q8_0: return (D % 32) ? -1 : (D / 32) * 34L;
    case FA_Q4_0: return (D % 32) ? -1 : (D / 32) * 18L;
  }
  return -1;
}

extern "C" size_t fab_workspace_size_capped(int N, int M, int H, int Hkv, int D, int Dv, size_t ws_cap) {
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv) return 0;
  int nsm = device_sms(nullptr, nullptr);
  if (nsm <= 0) nsm = 152;
  return make_plan(N, M, H, Hkv, D, Dv, nsm, ws_cap).total;
}

extern "C" size_t fa_back_workspace_size(int N, int M, int H, int Hkv, int D, int Dv) {
  return fab_workspace_size_capped(N, M, H, Hkv, D, Dv, SIZE_MAX);
}

extern "C" size_t fa_back_workspace_size_min(int N, int M, int H, int Hkv, int D, int Dv) {
  return fab_workspace_size_capped(N, M, H, Hkv, D, Dv, 0);
}

extern "C" fa_status fa_back_plan_info(int N, int M, int H, int Hkv, int D, int Dv, size_t workspace_bytes,
                                       int* level, int* key_splits, size_t* plan_bytes) {
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || Hkv > 256) return FA_ERR_SHAPE;
  if (!pick(D, Dv)) return FA_ERR_UNSUPPORTED;
  int nsm = device_sms(nullptr, nullptr);
  if (nsm <= 0) nsm = 152;  // no device: the GB300's SM count
  const Plan P = make_plan(N, M, H, Hkv, D, Dv, nsm, workspace_bytes);
  if (workspace_bytes < P.total) return FA_ERR_WORKSPACE;
  if (level) *level = P.dsq ? 2 : P.pre ? 1 : 0;
  if (key_splits) *key_splits = P.nsplit;
  if (plan_bytes) *plan_bytes = P.total;
  return FA_OK;
}

extern "C" fa_status fa_back(const float* q, const void* k, int k_type, const void* v, int v_type,
                             const uint16_t* mask, int mask_heads, const float* dO, float scale, int N, int M,
                             int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK, float* dV,
                             float* lse, float* delta, void* workspace, size_t workspace_bytes, void* stream) {
  // the plan is the fastest one whose workspace fits the caller's
  return fab_back_capped(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dQ,
                         dK, dV, lse, delta, workspace, workspace_bytes, stream, workspace_bytes, nullptr, nullptr,
                         nullptr);
}

extern "C" fa_status fa_back_batched(int B, const float* q, const void* k, int k_type, const void* v, int v_type,
                                     const uint16_t* mask, int mask_heads, int mask_per_batch, const float* dO,
                                     float scale, int N, int M, int H, int Hkv, int D, int Dv, int causal, float* dQ,
                                     float* dK, float* dV, float* lse, float* delta, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (B < 0) return FA_ERR_SHAPE;
  const long rbk = fa_row_bytes(k_type, D), rbv = fa_row_bytes(v_type, Dv);
  if (rbk <= 0 || rbv <= 0) return FA_ERR_SHAPE;
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0) return FA_ERR_SHAPE;
  const long hm = mask ? (mask_heads > 0 ? mask_heads : 1) : 0;
  // one problem after another on the stream, sharing the workspace; batch b's slices start
  // b problems into each tensor
  for (int b = 0; b < B; ++b) {
    const size_t nq = (size_t)b * N * H, nk = (size_t)b * M * Hkv;
    const fa_status rc = fa_back(
        q ? q + nq * D : nullptr, k ? static_cast<const uint8_t*>(k) + nk * rbk : nullptr, k_type,
        v ? static_cast<const uint8_t*>(v) + nk * rbv : nullptr, v_type,
        mask ? mask + (mask_per_batch ? (size_t)b * hm * N * M : 0) : nullptr, mask_heads, dO ? dO + nq * Dv : nullptr,
        scale, N, M, H, Hkv, D, Dv, causal, dQ ? dQ + nq * D : nullptr, dK ? dK + nk * D : nullptr,
        dV ? dV + nk * Dv : nullptr, lse ? lse + nq : nullptr, delta ? delta + nq : nullptr, workspace,
        workspace_bytes, stream);
    if (rc != FA_OK) return rc;
  }
  return FA_OK;
}

extern "C" size_t fa_forward_workspace_size(int N, int M, int H, int Hkv, int D, int Dv) {
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv) return 0;
  int nsm = device_sms(nullptr, nullptr);
  if (nsm <= 0) nsm = 152;
  return plan_variant(N, M, H, Hkv, D, Dv, nsm, SIZE_MAX, 1).total;
}

extern "C" fa_status fa_forward(const float* q, const void* k, int k_type, const void* v, int v_type,
                                const uint16_t* mask, int mask_heads, float scale, int N, int M, int H, int Hkv,
                                int D, int Dv, int causal, float* O, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (N > 0 && !O) return FA_ERR_NULL;
  if (O && (reinterpret_cast<uintptr_t>(O) & 15)) return FA_ERR_ALIGN;
  return fab_back_capped(q, k, k_type, v, v_type, mask, mask_heads, nullptr, scale, N, M, H, Hkv, D, Dv, causal,
                         nullptr, nullptr, nullptr, lse, nullptr, workspace, workspace_bytes, stream, SIZE_MAX,
                         nullptr, nullptr, O);
}

extern "C" fa_status fa_back_with_stats(const float* q, const void* k, int k_type, const void* v, int v_type,
                                        const uint16_t* mask, int mask_heads, const float* dO, const float* lse,
                                        const float* delta, float scale, int N, int M, int H, int Hkv, int D, int Dv,
                                        int causal, float* dQ, float* dK, float* dV, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (N > 0 && (!lse || !delta)) return FA_ERR_NULL;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 15)) || (delta && (reinterpret_cast<uintptr_t>(delta) & 15)))
    return FA_ERR_ALIGN;
  return fab_back_capped(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dQ,
                         dK, dV, nullptr, nullptr, workspace, workspace_bytes, stream, workspace_bytes, lse, delta,
                         nullptr);
}

extern "C" fa_status fab_back_capped(const float* q, const void* k, int k_type, const void* v, int v_type,
                                     const uint16_t* mask, int mask_heads, const float* dO, float scale, int N,
                                     int M, int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK,
                                     float* dV, float* lse, float* delta, void* workspace, size_t workspace_bytes,
                                     void* stream, size_t ws_cap, const float* lse_in, const float* delta_in,
                                     float* O) {
  const bool given = lse_in != nullptr;  // fa_back_with_stats: no lse/delta outputs
  const bool forward = O != nullptr;     // fa_forward: lse and O only
  // ---- argument checks (nothing is enqueued on failure)
  if (k_type < FA_F32 || k_type > FA_Q4_0 || v_type < FA_F32 || v_type > FA_Q4_0) return FA_ERR_TYPE;
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || Hkv > 256) return FA_ERR_SHAPE;
  if (mask && mask_heads != 1 && mask_heads != H) return FA_ERR_SHAPE;
  if (!pick(D, Dv)) return FA_ERR_UNSUPPORTED;
  if ((long)N * (H / Hkv) > (1L << 30) || M > (1 << 30)) return FA_ERR_UNSUPPORTED;
  const long rbk = fa_row_bytes(k_type, D), rbv = fa_row_bytes(v_type, Dv);
  if (rbk <= 0 || rbv <= 0) return FA_ERR_SHAPE;
  const bool needQ = N > 0, needK = M > 0;
  if (forward) {
    if (needQ && (!q || !lse || (needK && (!k || !v)))) return FA_ERR_NULL;
  } else if ((needQ && (!q || !dO || !dQ || (!given && (!lse || !delta)))) || (needK && (!k || !v || !dK || !dV))) {
    return FA_ERR_NULL;
  }
  const void* ptrs16[] = {q, dO, dQ, dK, dV, lse, delta, k, v, mask};
  for (const void* pp : ptrs16)
    if (pp && !aligned(pp, 16)) return FA_ERR_ALIGN;
  int major = 0, minor = 0;
  const int nsm = device_sms(&major, &minor);
  if (nsm <= 0) return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;
  // the forward runs plan level 1 (K'/V' copies, no stored dS)
  const Plan P = forward ? plan_variant(N, M, H, Hkv, D, Dv, nsm, SIZE_MAX, 1) : make_plan(N, M, H, Hkv, D, Dv, nsm, ws_cap);
  if (!workspace || workspace_bytes < P.total) return FA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // ---- degenerate shapes: every output element is still written
  if (N == 0 || M == 0) {
    const long nq = (long)N * H, nkd = (long)M * Hkv * D, nkv = (long)M * Hkv * Dv;
    auto fill = [&](float* x, long n, float val) {  // outputs the call does not have are null
      if (x && n > 0) k_fill<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, n, val);
    };
    fill(dK, nkd, 0.f);
    fill(dV, nkv, 0.f);
    if (lse) fill(lse, nq, -std::numeric_limits<float>::infinity());
    if (delta) fill(delta, nq, 0.f);
    if (O) fill(O, nq * Dv, 0.f);
    fill(dQ, nq * D, 0.f);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  int* errp = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&errp), g_err) != cudaSuccess) return FA_ERR_CUDA;

  Params p;
  std::memset(&p, 0, sizeof(p));
  p.q = q, p.dO = dO;
  p.k = reinterpret_cast<const uint8_t*>(k), p.v = reinterpret_cast<const uint8_t*>(v);
  p.k_type = k_type, p.v_type = v_type, p.rbk = (int)rbk, p.rbv = (int)rbv;
  p.mask = mask, p.Hm = mask ? mask_heads : 1;
  p.scale = scale;
  p.N = N, p.M = M, p.H = H, p.Hkv = Hkv, p.G = P.G, p.D = D, p.Dv = Dv, p.R = P.R, p.causal = causal ? 1 : 0;
  p.nQT = P.nQT, p.nKT = P.nKT, p.nsplit = P.nsplit, p.kt_per_split = P.kt_per_split;
  p.dQ = dQ, p.dK = dK, p.dV = dV, p.lse = lse, p.delta = delta;
  p.st = reinterpret_cast<Stats*>(ws + P.off_stats);
  p.rmean = reinterpret_cast<float*>(ws + P.off_rmean);
  p.dOr = reinterpret_cast<float*>(ws + P.off_dOr);
  p.lamr = reinterpret_cast<float*>(ws + P.off_lamr);
  p.lse2 = reinterpret_cast<float*>(ws + P.off_lse2);
  p.dlt = reinterpret_cast<float*>(ws + P.off_dlt);
  p.part = reinterpret_cast<float*>(ws + P.off_part);
  p.dqpart = reinterpret_cast<float*>(ws + P.off_dqpart);
  p.q16 = reinterpret_cast<__half*>(ws + P.off_q16);
  p.do16 = reinterpret_cast<__half*>(ws + P.off_do16);
  p.bstat = reinterpret_cast<float*>(ws + P.off_bstat);
  p.nblk_stats = P.nblk_stats;
  p.vsum = reinterpret_cast<float*>(ws + P.off_vsum);
  p.nbv = P.nbv;
  p.rsh = reinterpret_cast<float*>(ws + P.off_rsh);
  p.kd = P.pre ? reinterpret_cast<__half*>(ws + P.off_kd) : nullptr;
  p.vd = P.pre ? reinterpret_cast<__half*>(ws + P.off_vd) : nullptr;
  p.ds = P.dsq ? reinterpret_cast<__half*>(ws + P.off_ds) : nullptr;
  p.ldds = P.ldds;
  p.lse_in = lse_in, p.delta_in = delta_in;
  p.o_out = O;
  p.raw_bulk = (rbk % 16 == 0 && rbv % 16 == 0 && rbk <= 2048 && rbv <= 2048) ? 1 : 0;
  p.rbk_pad = (int)((rbk + 15) / 16 * 16);
  p.rbv_pad = (int)((rbv + 15) / 16 * 16);
  p.err = errp;

  CUtensorMap tmQ, tmO;
  if (!make_map(&tmQ, p.q16, D, P.R, Hkv) || !make_map(&tmO, p.do16, Dv, P.R, Hkv)) return FA_ERR_CUDA;

  CallRec rec;
  rec.begin(s);
  k_row_stats<<<P.nblk_stats, 256, 0, s>>>(p);
  rec.mark(KS_STATS);
  k_vsum<<<(unsigned)(P.nbv * Hkv), 256, 0, s>>>(p);
  rec.mark(KS_VSUM);
  k_finalize<<<1, 1024, 0, s>>>(p);
  rec.mark(KS_FINAL);
  k_convert<<<(unsigned)std::min<long>(((long)N * H + 7) / 8, 8L * nsm), 256, 0, s>>>(p);
  rec.mark(KS_CONVERT);
  if (given) {
    k_stats_in<<<(unsigned)(((long)Hkv * P.R + 255) / 256), 256, 0, s>>>(p);
    rec.mark(KS_STATS_IN);
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  return (forward ? pick_fwd(D, Dv) : pick(D, Dv))(p, P, tmQ, tmO, s, rec) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_back_selftest_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return FA_ERR_SHAPE;
  int* errp = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&errp), g_err) != cudaSuccess) return FA_ERR_CUDA;
  k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(errp, limit_ns);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_back_get_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return v ? (fa_status)v : FA_OK;
}

extern "C" const char* fa_back_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_TYPE: return "unknown K or V cache type";
    case FA_ERR_SHAPE: return "invalid shape (H % Hkv, mask heads, or a format's block size)";
    case FA_ERR_ALIGN: return "misaligned pointer";
    case FA_ERR_UNSUPPORTED: return "unsupported head size or problem size";
    case FA_ERR_DEVICE: return "the current device is not sm_103";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

extern "C" fa_status fa_back_profile(int enable) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.on = enable != 0;
  return FA_OK;
}

extern "C" int fa_back_profile_read(float* ms_sum, int* launches, const char** names, int max_kernels) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  const int n = std::min(max_kernels, (int)KS_N);
  for (int k = 0; k < n; ++k) {
    if (ms_sum) ms_sum[k] = 0.f;
    if (launches) launches[k] = 0;
    if (names) names[k] = kKernelNames[k];
  }
  for (int c = 0; c < g_prof.ncalls; ++c) {
    int prev = kProfSlots;  // start marker
    for (int m = 0; m < g_prof.nmarks[c]; ++m) {
      const int k = g_prof.order[c][m];
      float ms = 0.f;
      if (cudaEventSynchronize(g_prof.ev[c][k]) == cudaSuccess &&
          cudaEventElapsedTime(&ms, g_prof.ev[c][prev], g_prof.ev[c][k]) == cudaSuccess && k < n) {
        if (ms_sum) ms_sum[k] += ms;
        if (launches) launches[k] += 1;
      }
      prev = k;
    }
  }
  g_prof.ncalls = 0;
  return n;
}
