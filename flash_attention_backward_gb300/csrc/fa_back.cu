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
#include <atomic>
#include <cmath>
#include <cstring>
#include <limits>
#include <mutex>

#include "../../include/fa_back.h"
#include "fa_internal.h"
#include "fa_launch.cuh"


namespace fab {

__device__ int g_err = 0;


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
  P.off_sg = o; o = align256(o + sizeof(float) * (size_t)Hkv * P.R);  // per-row sink-gradient terms
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

// Launch plan and workspace layout for one variant (level 2: binary16 K'/V' copies and the stored
// dS with a dQ product over it; 3: the stored dS without the copies, every pass decoding the raw
// cache; 1: the copies only, feeding the row passes; 0: passes decoding the raw cache).  The
// keys of each row tile are split so that the last wave of CTAs (one per SM) wastes least,
// counting a small cost per split for the partial merges; among split counts whose workspace
// fits `ws_cap`, the cheapest is taken (1 if none fits).
static Plan plan_variant(int N, int M, int H, int Hkv, int D, int Dv, int nsm, size_t ws_cap, int level) {
  Plan P;
  std::memset(&P, 0, sizeof(P));
  P.pre = level == 1 || level == 2;
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

// The fastest plan whose workspace fits ws_cap, trying the levels in the order of their speed
// (2, 3, 1; their workspaces grow as 1 < 3 < 2); level 0 with one split is the smallest workspace
// fa_back() accepts.  nocopy keeps to the plans without the binary16 copy of the cache (3, 0).
static Plan make_plan(int N, int M, int H, int Hkv, int D, int Dv, int nsm, size_t ws_cap = SIZE_MAX,
                      bool nocopy = false) {
  static const int kOrder[] = {2, 3, 1};
  for (int level : kOrder) {
    if (nocopy && level != 3) continue;
    const Plan P = plan_variant(N, M, H, Hkv, D, Dv, nsm, ws_cap, level);
    if (P.total <= ws_cap) return P;
  }
  return plan_variant(N, M, H, Hkv, D, Dv, nsm, ws_cap, 0);
}

static int plan_level(const Plan& P) { return P.dsq ? (P.pre ? 2 : 3) : P.pre ? 1 : 0; }

static int device_sms(int* major, int* minor) {
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (major) cudaDeviceGetAttribute(major, cudaDevAttrComputeCapabilityMajor, dev);
  if (minor) cudaDeviceGetAttribute(minor, cudaDevAttrComputeCapabilityMinor, dev);
  return nsm;
}


// ------------------------------------------------------------------------------------------------
// measurement hook: one CUDA event before the sequence and one after each launch

// (the read-out measures each kernel from the marker recorded before it)
static const char* const kKernelNames[kProfSlots] = {
    "k_row_stats", "k_vsum", "k_finalize", "k_convert", "k_predecode", "k_rows_lse", "k_lse_merge", "k_rows_dq",
    "k_dq_reduce", "k_cols", "k_dq_gemm", "k_stats_in", "k_fwd", "k_fwd_merge", "k_cols_rowscale", "k_sink_grad",
    "k_dq_raw"};
Profiler g_prof;

// Failure-detection hook: the wait limit of the next call's kernels plus one (0: none pending).
static std::atomic<unsigned long long> g_next_wait_ns{0};

static RunFn pick_seq(int D, int Dv, bool ext, bool forward) {
  switch (D) {
    case 64: return ext && !forward ? pick_d64_ext(Dv) : pick_d64(Dv, forward);
    case 128: return ext && !forward ? pick_d128_ext(Dv) : pick_d128(Dv, forward);
    case 256: return ext && !forward ? pick_d256_ext(Dv) : pick_d256(Dv, forward);
  }
  return nullptr;
}
static RunFn pick(int D, int Dv) { return pick_seq(D, Dv, false, false); }

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

extern "C" size_t fa_back_workspace_size_nocopy(int N, int M, int H, int Hkv, int D, int Dv) {
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv) return 0;
  int nsm = device_sms(nullptr, nullptr);
  if (nsm <= 0) nsm = 152;
  return make_plan(N, M, H, Hkv, D, Dv, nsm, SIZE_MAX, true).total;
}

extern "C" fa_status fa_back_plan_info(int N, int M, int H, int Hkv, int D, int Dv, size_t workspace_bytes,
                                       int* level, int* key_splits, size_t* plan_bytes) {
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || Hkv > 256) return FA_ERR_SHAPE;
  if (!pick(D, Dv)) return FA_ERR_UNSUPPORTED;
  int nsm = device_sms(nullptr, nullptr);
  if (nsm <= 0) nsm = 152;  // no device: the GB300's SM count
  const Plan P = make_plan(N, M, H, Hkv, D, Dv, nsm, workspace_bytes);
  if (workspace_bytes < P.total) return FA_ERR_WORKSPACE;
  if (level) *level = plan_level(P);
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
                         nullptr, nullptr);
}

extern "C" fa_status fa_back_ext(const float* q, const void* k, int k_type, const void* v, int v_type,
                                 const uint16_t* mask, int mask_heads, const float* dO, float scale, int N, int M,
                                 int H, int Hkv, int D, int Dv, int causal, const float* alibi_slopes, float softcap,
                                 const float* sinks, float* dsinks, float* dQ, float* dK, float* dV, float* lse,
                                 float* delta, void* workspace, size_t workspace_bytes, void* stream) {
  const fab_opts x = {alibi_slopes, softcap, sinks, dsinks, 0};
  return fab_back_capped(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dQ,
                         dK, dV, lse, delta, workspace, workspace_bytes, stream, workspace_bytes, nullptr, nullptr,
                         nullptr, &x);
}

extern "C" fa_status fa_back_nocopy(const float* q, const void* k, int k_type, const void* v, int v_type,
                                    const uint16_t* mask, int mask_heads, const float* dO, float scale, int N, int M,
                                    int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK, float* dV,
                                    float* lse, float* delta, void* workspace, size_t workspace_bytes, void* stream) {
  const fab_opts x = {nullptr, 0.f, nullptr, nullptr, 1};
  return fab_back_capped(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dQ,
                         dK, dV, lse, delta, workspace, workspace_bytes, stream, workspace_bytes, nullptr, nullptr,
                         nullptr, &x);
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
                         nullptr, nullptr, O, nullptr);
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
                         nullptr, nullptr);
}

extern "C" fa_status fab_back_capped(const float* q, const void* k, int k_type, const void* v, int v_type,
                                     const uint16_t* mask, int mask_heads, const float* dO, float scale, int N,
                                     int M, int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK,
                                     float* dV, float* lse, float* delta, void* workspace, size_t workspace_bytes,
                                     void* stream, size_t ws_cap, const float* lse_in, const float* delta_in,
                                     float* O, const fab_opts* ext) {
  const bool given = lse_in != nullptr;  // fa_back_with_stats: no lse/delta outputs
  const bool forward = O != nullptr;     // fa_forward: lse and O only
  const fab_opts none = {nullptr, 0.f, nullptr, nullptr, 0};
  const fab_opts& X = ext ? *ext : none;
  if (!(X.softcap >= 0.f) || !std::isfinite(X.softcap)) return FA_ERR_SHAPE;
  if ((given || forward) && (X.alibi || X.softcap > 0.f || X.sinks)) return FA_ERR_UNSUPPORTED;
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
  const void* ptrs4[] = {X.alibi, X.sinks, X.sinks ? X.dsinks : nullptr};
  for (const void* pp : ptrs4)
    if (pp && !aligned(pp, 4)) return FA_ERR_ALIGN;
  int major = 0, minor = 0;
  const int nsm = device_sms(&major, &minor);
  if (nsm <= 0) return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;
  // the forward runs plan level 1 (K'/V' copies, no stored dS)
  const Plan P = forward ? plan_variant(N, M, H, Hkv, D, Dv, nsm, SIZE_MAX, 1)
                         : make_plan(N, M, H, Hkv, D, Dv, nsm, ws_cap, X.nocopy != 0);
  if (!workspace || workspace_bytes < P.total) return FA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned long long wait_hook = g_next_wait_ns.exchange(0);  // this call takes a pending limit

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
    if (X.sinks) {  // rows hold the sink alone (or there are no rows): lse = sigma, dsinks = 0
      const long n = std::max<long>(nq, H);
      k_sink_only<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(X.sinks, M == 0 ? lse : nullptr, delta, X.dsinks, M == 0 ? N : 0, H);
    }
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
  p.wait_ns = wait_hook ? wait_hook - 1 : kWaitLimitNs;
  p.softcap = X.softcap;
  p.alibi = X.alibi;
  p.sinks = X.sinks;
  p.dsinks = X.sinks ? X.dsinks : nullptr;
  p.sg = p.dsinks ? reinterpret_cast<float*>(ws + P.off_sg) : nullptr;

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
  const bool scores_ext = p.alibi != nullptr || p.softcap > 0.f;  // the EXT kernels form the scores
  return pick_seq(D, Dv, scores_ext, forward)(p, P, tmQ, tmO, s, rec) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_back_selftest_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return FA_ERR_SHAPE;
  int* errp = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&errp), g_err) != cudaSuccess) return FA_ERR_CUDA;
  k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(errp, limit_ns);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_back_test_wait_limit(unsigned long long limit_ns) {
  if (limit_ns > kWaitLimitNs) return FA_ERR_SHAPE;
  g_next_wait_ns.store(limit_ns + 1);
  return FA_OK;
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
