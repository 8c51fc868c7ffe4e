// Device code of the flash-attention backward over a raw K/V cache (sm_103a).
//
// Pipeline (all on one stream, see fa_back.cu):
//   k_row_stats  -> per-block max |x| and max row norm of Q, dO, K^ and V^
//   k_vsum       -> per-chunk column sums of V^ (for its column mean r)
//   k_finalize   -> power-of-two operand scales, r, the dS multiplier
//   k_convert    -> Q, dO as scaled binary16 rows packed per KV head (row r = i*G + g)
//   k_rows<LSE>  -> per (row tile, key split): running max / sum / sum of p*dP
//   k_lse_merge  -> lse, delta outputs; log2-domain lse and shifted delta for the gradient passes
//   k_rows<DQ>   -> dQ = scale * dS K^ per row tile (split over keys, merged in fixed order)
//   k_cols       -> dK^T = scale * Q^T dS and dV^T = dO^T P per key tile
//
// Arithmetic (documented in the header of fa_back.cu): every tensor-core product is
// binary16 x binary16 -> f32 (tcgen05.mma kind::f16).  Inputs are multiplied by powers of two
// so that their largest magnitude sits near 2^14, which keeps them in binary16's normal range
// without changing any product.  V is shifted by its per-column mean r before rounding: softmax
// rows sum to one, so dP_ij - delta_i is unchanged by the shift while the rounded operand
// keeps the relative precision of V's variation (the near-constant-V case).
#pragma once
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "sm100.cuh"

namespace fab {

constexpr int kTypeF32 = 0, kTypeF16 = 1, kTypeQ8 = 2, kTypeQ4 = 3;
constexpr int kErrTimeout = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Scales and factors shared by every kernel after k_finalize (workspace resident).
struct Stats {
  float sQ, sK, sdO, sV;  // operand scales (powers of two)
  float lam;              // dS multiplier (power of two)
  float sP;               // P multiplier (2^15)
  float c2;               // scale * log2(e) / (sQ * sK): maps the Q.K accumulator to log2 units
  float dq_fac, dk_fac, dv_fac, delta_fac;
  float amax[4], norm2[4];
  float rnorm, ramax;
};

struct Params {
  const float* q;
  const float* dO;
  const uint8_t* k;
  const uint8_t* v;
  int k_type, v_type, rbk, rbv;
  const uint16_t* mask;
  int Hm;
  float scale;
  int N, M, H, Hkv, G, D, Dv, R, causal;
  int nQT, nKT, nsplit, kt_per_split;
  float* dQ;
  float* dK;
  float* dV;
  float* lse;
  float* delta;
  // workspace
  Stats* st;
  float* rmean;   // [Hkv][Dv]
  float* dOr;     // [Hkv][R]   dO_i . r
  float* lse2;    // [Hkv][R]   lse / ln 2 (or -inf)
  float* dlt;     // [Hkv][R]   shifted delta in accumulator units
  float* part;    // [nsplit][Hkv][R][3]
  float* dqpart;  // [nsplit][Hkv][R][D]
  __half* q16;    // [Hkv][R][D]
  __half* do16;   // [Hkv][R][Dv]
  float* bstat;   // [nblk_stats][4][2]
  int nblk_stats;
  float* vsum;    // [nbv][Hkv][Dv]
  int nbv;
  int* err;
};

__host__ __device__ constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

// ------------------------------------------------------------------------------------------------
// decoding raw cache rows

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Scalar decode of element c of a raw row (used by the statistics passes).
__device__ __forceinline__ float decode_elem(const uint8_t* row, int type, int c) {
  if (type == kTypeF32) return __ldg(reinterpret_cast<const float*>(row) + c);
  if (type == kTypeF16) return h2f(__ldg(reinterpret_cast<const unsigned short*>(row) + c));
  if (type == kTypeQ8) {
    const uint8_t* b = row + 34 * (c >> 5);
    const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
    return (float)(int8_t)__ldg(b + 2 + (c & 31)) * d;
  }
  const uint8_t* b = row + 18 * (c >> 5);
  const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
  const int o = c & 31;
  const uint8_t byte = __ldg(b + 2 + (o & 15));
  const int nib = o < 16 ? (byte & 15) : (byte >> 4);
  return (float)(nib - 8) * d;
}

// Decode 8 consecutive elements c0..c0+7 (c0 % 8 == 0) of a raw row; the codes are unpacked in
// pairs and every value is exact in f32 (a q8_0 value has at most 7 + 11 significant bits).
__device__ __forceinline__ void decode8(const uint8_t* row, int type, int c0, float* x) {
  if (type == kTypeF32) {
    const float4* p = reinterpret_cast<const float4*>(row + 4 * c0);
    const float4 a = __ldg(p), b = __ldg(p + 1);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
  } else if (type == kTypeF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + 2 * c0));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      x[2 * e] = f.x, x[2 * e + 1] = f.y;
    }
  } else if (type == kTypeQ8) {
    const uint8_t* b = row + 34 * (c0 >> 5);
    const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
    const unsigned short* cp = reinterpret_cast<const unsigned short*>(b + 2 + (c0 & 31));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const unsigned short pr = __ldg(cp + e);  // two codes
      x[2 * e] = (float)(int8_t)(pr & 0xff) * d;
      x[2 * e + 1] = (float)(int8_t)(pr >> 8) * d;
    }
  } else {
    const uint8_t* b = row + 18 * (c0 >> 5);
    const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
    const int o = c0 & 31;
    const unsigned short* cp = reinterpret_cast<const unsigned short*>(b + 2 + (o & 15));
    const int sh = o < 16 ? 0 : 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const unsigned short pr = __ldg(cp + e);  // two bytes -> two nibbles of this half
      x[2 * e] = (float)((int)((pr >> sh) & 15) - 8) * d;
      x[2 * e + 1] = (float)((int)((pr >> (8 + sh)) & 15) - 8) * d;
    }
  }
}

// Decode BK cache rows (keys j0.., KV head hk) into a binary16 operand tile: DD/64 panels of
// [BK rows][64 columns], 128-byte rows, 128-byte swizzled.  Keys >= M become zero rows.
// out = (x^ - shift[c]) * sigma  (shift may be null).
template <int DD, int BK, int NT>
__device__ __forceinline__ void decode_tile(const uint8_t* base, int type, int rb, int hk, int Hkv, int j0, int M,
                                            uint8_t* panels, float sigma, const float* shift) {
  constexpr int UPR = DD / 8;  // 8-element units per row
  for (int u = threadIdx.x; u < BK * UPR; u += NT) {
    const int row = u / UPR;
    const int c0 = (u % UPR) * 8;
    const int j = j0 + row;
    float x[8];
    if (j < M) {
      decode8(base + ((size_t)j * Hkv + hk) * rb, type, c0, x);
      if (shift) {
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(shift + c0));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(shift + c0 + 4));
        x[0] -= s0.x, x[1] -= s0.y, x[2] -= s0.z, x[3] -= s0.w;
        x[4] -= s1.x, x[5] -= s1.y, x[6] -= s1.z, x[7] -= s1.w;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= sigma;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
    }
    uint4 w;
    __half2 h0 = __floats2half2_rn(x[0], x[1]), h1 = __floats2half2_rn(x[2], x[3]);
    __half2 h2 = __floats2half2_rn(x[4], x[5]), h3 = __floats2half2_rn(x[6], x[7]);
    w.x = *reinterpret_cast<uint32_t*>(&h0), w.y = *reinterpret_cast<uint32_t*>(&h1);
    w.z = *reinterpret_cast<uint32_t*>(&h2), w.w = *reinterpret_cast<uint32_t*>(&h3);
    const uint32_t off = (uint32_t)(c0 / 64) * (BK * 128) + swz128((uint32_t)row * 128 + (uint32_t)((c0 & 63) / 8) * 16);
    *reinterpret_cast<uint4*>(panels + off) = w;
  }
}

// Store 32 binary16 values (one row, columns col0..col0+31 of a [128][BK] panel set).
template <int BK>
__device__ __forceinline__ void store_row32(uint8_t* panels, int row, int col0, const float* v, float mul) {
  const uint32_t pbase = (uint32_t)(col0 / 64) * (128 * 128);
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __half2 hh = __floats2half2_rn(v[q4 * 8 + 2 * e] * mul, v[q4 * 8 + 2 * e + 1] * mul);
      wp[e] = *reinterpret_cast<uint32_t*>(&hh);
    }
    const int col = (col0 & 63) + q4 * 8;
    *reinterpret_cast<uint4*>(panels + pbase + swz128((uint32_t)row * 128 + (uint32_t)(col / 8) * 16)) = w;
  }
}

__device__ __forceinline__ void record_error(int* err, int code) { atomicExch(err, code); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ------------------------------------------------------------------------------------------------
// statistics and packing

// One warp per row of Q, dO, K^ or V^: max |x| and max squared row norm, reduced per block.
__global__ void __launch_bounds__(256) k_row_stats(Params p) {
  __shared__ float red[8][4][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long nQ = (long)p.N * p.H, nK = (long)p.M * p.Hkv;
  const long tot = 2 * nQ + 2 * nK;
  float amax[4] = {0, 0, 0, 0}, nrm[4] = {0, 0, 0, 0};
  for (long rw = (long)blockIdx.x * 8 + warp; rw < tot; rw += (long)gridDim.x * 8) {
    int t;
    long r;
    if (rw < nQ) t = 0, r = rw;
    else if (rw < 2 * nQ) t = 1, r = rw - nQ;
    else if (rw < 2 * nQ + nK) t = 2, r = rw - 2 * nQ;
    else t = 3, r = rw - 2 * nQ - nK;
    const int DD = (t == 0 || t == 2) ? p.D : p.Dv;
    float am = 0.f, ss = 0.f;
    for (int c = lane; c < DD; c += 32) {
      float x;
      if (t == 0) x = __ldg(p.q + r * p.D + c);
      else if (t == 1) x = __ldg(p.dO + r * p.Dv + c);
      else if (t == 2) x = decode_elem(p.k + r * p.rbk, p.k_type, c);
      else x = decode_elem(p.v + r * p.rbv, p.v_type, c);
      am = fmaxf(am, fabsf(x));
      ss = fmaf(x, x, ss);
    }
    am = warp_max(am);
    ss = warp_sum(ss);
    amax[t] = fmaxf(amax[t], am);
    nrm[t] = fmaxf(nrm[t], ss);
  }
  if (lane == 0)
    for (int t = 0; t < 4; ++t) red[warp][t][0] = amax[t], red[warp][t][1] = nrm[t];
  __syncthreads();
  if (threadIdx.x < 8) {
    const int t = threadIdx.x >> 1, w = threadIdx.x & 1;
    float m = 0.f;
    for (int k = 0; k < 8; ++k) m = fmaxf(m, red[k][t][w]);
    p.bstat[((size_t)blockIdx.x * 4 + t) * 2 + w] = m;
  }
}

// Column sums of V^ over a chunk of keys; thread = (hk, c); keys summed in increasing order.
__global__ void __launch_bounds__(256) k_vsum(Params p) {
  const int idx = blockIdx.x * 256 + threadIdx.x;
  if (idx >= p.Hkv * p.Dv) return;
  const int hk = idx / p.Dv, c = idx % p.Dv;
  const long per = ((long)p.M + p.nbv - 1) / p.nbv;
  const long ja = (long)blockIdx.y * per, jb = min((long)p.M, ja + per);
  float s = 0.f;
  for (long j = ja; j < jb; ++j) s += decode_elem(p.v + (j * p.Hkv + hk) * p.rbv, p.v_type, c);
  p.vsum[((size_t)blockIdx.y * p.Hkv + hk) * p.Dv + c] = s;
}

__device__ __forceinline__ float pow2_scale_for(float amax, int target_exp) {
  // 2^(target - e) where amax < 2^e, so amax * scale < 2^target; 1 for an all-zero tensor.
  if (!(amax > 0.f) || !isfinite(amax)) return 1.f;
  int e;
  frexpf(amax, &e);
  int s = target_exp - e;
  s = max(-120, min(120, s));
  return ldexpf(1.f, s);
}

__global__ void __launch_bounds__(256) k_finalize(Params p) {
  __shared__ float am[4], nm[4];
  __shared__ float rn2[1024], ram[1024];
  const int tid = threadIdx.x;
  if (tid < 8) {
    const int t = tid >> 1, w = tid & 1;
    float m = 0.f;
    for (int b = 0; b < p.nblk_stats; ++b) m = fmaxf(m, p.bstat[((size_t)b * 4 + t) * 2 + w]);
    if (w == 0) am[t] = m;
    else nm[t] = m;
  }
  // column means of V^ (chunks in order), per-head squared norm and max |r|
  float my_am = 0.f;
  const float invM = p.M > 0 ? 1.f / (float)p.M : 0.f;
  for (int idx = tid; idx < p.Hkv * p.Dv; idx += 256) {
    float s = 0.f;
    for (int b = 0; b < p.nbv; ++b) s += p.vsum[((size_t)b * p.Hkv) * p.Dv + idx];
    const float r = s * invM;
    p.rmean[idx] = r;
    my_am = fmaxf(my_am, fabsf(r));
  }
  __syncthreads();
  // squared norm of each head's r, taken in a fixed order by one thread per head
  if (tid < p.Hkv && tid < 1024) {
    float n2 = 0.f;
    for (int c = 0; c < p.Dv; ++c) n2 = fmaf(p.rmean[tid * p.Dv + c], p.rmean[tid * p.Dv + c], n2);
    rn2[tid] = n2;
  }
  ram[tid] = my_am;
  __syncthreads();
  if (tid == 0) {
    float rmax2 = 0.f, ramax = 0.f;
    for (int h = 0; h < p.Hkv && h < 1024; ++h) rmax2 = fmaxf(rmax2, rn2[h]);
    for (int t = 0; t < 256; ++t) ramax = fmaxf(ramax, ram[t]);
    Stats s;
    for (int t = 0; t < 4; ++t) s.amax[t] = am[t], s.norm2[t] = nm[t];
    s.rnorm = sqrtf(rmax2);
    s.ramax = ramax;
    s.sQ = pow2_scale_for(am[0], 14);
    s.sdO = pow2_scale_for(am[1], 14);
    s.sK = pow2_scale_for(am[2], 14);
    const float vamax = am[3] + ramax;  // |v^ - r| <= |v^| + |r|
    s.sV = pow2_scale_for(vamax, 14);
    s.sP = 32768.f;
    // |dP'_ij - delta'_i| <= 2 max_j |dO_i . (v^_j - r)| <= 2 |dO_i| (|v^_j| + |r|), in scaled units
    const float bound = 2.f * (sqrtf(nm[1]) * s.sdO) * ((sqrtf(nm[3]) + s.rnorm) * s.sV) * 1.0001f;
    s.lam = pow2_scale_for(bound, 15);
    s.c2 = p.scale * kLog2e / (s.sQ * s.sK);
    s.dq_fac = p.scale / (s.lam * s.sdO * s.sV * s.sK);
    s.dk_fac = p.scale / (s.lam * s.sdO * s.sV * s.sQ);
    s.dv_fac = 1.f / (s.sP * s.sdO);
    s.delta_fac = 1.f / (s.sdO * s.sV);
    *p.st = s;
  }
}

// One warp per (i, h): binary16 rows of Q and dO (row r = i*G + g of head hk) and dO_i . r.
__global__ void __launch_bounds__(256) k_convert(Params p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long nrow = (long)p.N * p.H;
  const float sQ = p.st->sQ, sdO = p.st->sdO;
  for (long rw = (long)blockIdx.x * 8 + warp; rw < nrow; rw += (long)gridDim.x * 8) {
    const int i = (int)(rw / p.H), h = (int)(rw % p.H);
    const int hk = h / p.G, g = h % p.G;
    const long r = (long)i * p.G + g;
    const float* qs = p.q + rw * p.D;
    __half* qd = p.q16 + ((size_t)hk * p.R + r) * p.D;
    for (int c = 2 * lane; c < p.D; c += 64) {
      const float2 x = __ldg(reinterpret_cast<const float2*>(qs + c));
      *reinterpret_cast<__half2*>(qd + c) = __floats2half2_rn(x.x * sQ, x.y * sQ);
    }
    const float* os = p.dO + rw * p.Dv;
    __half* od = p.do16 + ((size_t)hk * p.R + r) * p.Dv;
    const float* rm = p.rmean + (size_t)hk * p.Dv;
    float dot = 0.f;
    for (int c = 2 * lane; c < p.Dv; c += 64) {
      const float2 x = __ldg(reinterpret_cast<const float2*>(os + c));
      *reinterpret_cast<__half2*>(od + c) = __floats2half2_rn(x.x * sdO, x.y * sdO);
      dot = fmaf(x.x, rm[c], dot);
      dot = fmaf(x.y, rm[c + 1], dot);
    }
    dot = warp_sum(dot);
    if (lane == 0) p.dOr[(size_t)hk * p.R + r] = dot;
  }
}

// ------------------------------------------------------------------------------------------------
// row-tile passes: LSE/D statistics (MODE 0) and dQ (MODE 1)

template <int D, int Dv, int BK, int MODE>
struct RowsCfg {
  static constexpr int QB = 128 * D * 2, OB = 128 * Dv * 2, KB = BK * D * 2, VB = BK * Dv * 2;
  static constexpr int SB = MODE ? 128 * BK * 2 : 0;
  static constexpr int OFF_Q = 0, OFF_O = QB, OFF_K = QB + OB, OFF_V = OFF_K + KB, OFF_S = OFF_V + VB;
  static constexpr int OFF_BAR = OFF_S + SB;
  static constexpr int SMEM = OFF_BAR + 64 + 1024;  // + alignment slack
  static constexpr int TCOLS = pow2_at_least(MODE ? 2 * BK + D : 2 * BK);
};

template <int D, int Dv, int BK, int MODE>
__global__ void __launch_bounds__(128, 1)
    k_rows(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO, Params p) {
  using C = RowsCfg<D, Dv, BK, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sO = sm + C::OFF_O;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sS = sm + C::OFF_S;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 16);
  int* s_abort = reinterpret_cast<int*>(sm + C::OFF_BAR + 20);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int r0 = qt * 128;
  const int R = p.R, G = p.G;

  int kt_begin = split * p.kt_per_split;
  int kt_end = min(p.nKT, kt_begin + p.kt_per_split);
  if (p.causal) {
    const long i_hi = (long)min(R - 1, r0 + 127) / G;
    const long jmax = (long)p.M - p.N + i_hi;
    const int ntv = jmax < 0 ? 0 : (int)(jmax / BK) + 1;
    kt_end = min(kt_end, ntv);
  }

  if (warp == 0) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    *s_abort = 0;
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase, tP = tbase + BK, tAcc = tbase + 2 * BK;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  const Stats st = *p.st;
  // this thread's row
  const int r = r0 + tid;
  const bool rvalid = r < R;
  const int i = rvalid ? r / G : 0;
  const int h = hk * G + (rvalid ? r % G : 0);
  const long jlast = rvalid ? (p.causal ? min((long)p.M - 1, (long)p.M - p.N + i) : (long)p.M - 1) : -1;
  const uint16_t* mrow = p.mask ? p.mask + ((size_t)(h % p.Hm) * p.N + i) * p.M : nullptr;
  float lse2 = -CUDART_INF_F, dl = 0.f;
  if (MODE == 1 && rvalid) {
    lse2 = p.lse2[(size_t)hk * R + r];
    dl = p.dlt[(size_t)hk * R + r];
  }
  const bool live = MODE == 1 ? (lse2 > -CUDART_INF_F) : rvalid;
  float m2 = -CUDART_INF_F, l = 0.f, lc = 0.f, sd = 0.f, sdc = 0.f;

  bool have_tiles = kt_begin < kt_end;
  if (have_tiles && tid == 0) {
    mbar_arrive_expect_tx(&bars[0], (uint32_t)(C::QB + C::OB));
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * 128 * 128, &tmQ, &bars[0], c * 64, r0, hk);
#pragma unroll
    for (int c = 0; c < Dv / 64; ++c) tma_load_3d(sO + c * 128 * 128, &tmO, &bars[0], c * 64, r0, hk);
  }
  if (have_tiles) {
    if (!mbar_wait_bounded(&bars[0], 0, kWaitLimitNs)) {
      *s_abort = 1;
      record_error(p.err, kErrTimeout);
    }
  }
  __syncthreads();
  if (*s_abort) have_tiles = false;

  constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
  constexpr uint32_t ID_DQ = idesc_f16(128, D, false, true);
  uint32_t mma_phase = 0;
  bool first = true;
  const float* vshift = p.rmean + (size_t)hk * Dv;

  for (int kt = kt_begin; have_tiles && kt < kt_end; ++kt) {
    const int j0 = kt * BK;
    decode_tile<D, BK, 128>(p.k, p.k_type, p.rbk, hk, p.Hkv, j0, p.M, sK, st.sK, nullptr);
    decode_tile<Dv, BK, 128>(p.v, p.v_type, p.rbv, hk, p.Hkv, j0, p.M, sV, st.sV, vshift);
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t aq = smem_u32(sQ), ao = smem_u32(sO), bk = smem_u32(sK), bv = smem_u32(sV);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_f16(tS, sdesc_sw128(aq + (k / 4) * (128 * 128) + (k % 4) * 32, 16, 1024),
                sdesc_sw128(bk + (k / 4) * (BK * 128) + (k % 4) * 32, 16, 1024), ID_S, k > 0);
#pragma unroll
      for (int k = 0; k < Dv / 16; ++k)
        mma_f16(tP, sdesc_sw128(ao + (k / 4) * (128 * 128) + (k % 4) * 32, 16, 1024),
                sdesc_sw128(bv + (k / 4) * (BK * 128) + (k % 4) * 32, 16, 1024), ID_S, k > 0);
      mma_commit(&bars[1]);
    }
    if (!mbar_wait_bounded(&bars[1], mma_phase, kWaitLimitNs)) {
      *s_abort = 1;
      record_error(p.err, kErrTimeout);
    }
    mma_phase ^= 1;
    tc_fence_after();

#pragma unroll 1
    for (int c32 = 0; c32 < BK / 32; ++c32) {
      float s[32], dp[32];
      tmem_ld32(tS + lane_off + c32 * 32, s);
      tmem_ld32(tP + lane_off + c32 * 32, dp);
      tmem_ld_wait();
      const int jb = j0 + c32 * 32;
      float t2[32];
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        const int j = jb + n;
        bool ok = (long)j <= jlast;
        float mv = 0.f;
        if (ok && mrow) {
          mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
          ok = !(mv == -CUDART_INF_F);
        }
        t2[n] = ok ? fmaf(s[n], st.c2, mv * kLog2e) : -CUDART_INF_F;
      }
      if (MODE == 0) {
        float cmax = -CUDART_INF_F;
#pragma unroll
        for (int n = 0; n < 32; ++n) cmax = fmaxf(cmax, t2[n]);
        if (cmax > m2) {
          const float f = exp2f(m2 - cmax);  // 0 when m2 = -inf
          l *= f, lc *= f, sd *= f, sdc *= f;
          m2 = cmax;
        }
        if (cmax > -CUDART_INF_F) {
          float cl = 0.f, cs = 0.f;
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            const float e = exp2f(t2[n] - m2);  // 0 for masked keys
            cl += e;
            cs = fmaf(e, dp[n], cs);
          }
          // compensated accumulation of the chunk sums
          float y = cl - lc, t = l + y;
          lc = (t - l) - y, l = t;
          y = cs - sdc, t = sd + y;
          sdc = (t - sd) - y, sd = t;
        }
      } else {
        float ds[32];
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          const float pr = (live && t2[n] > -CUDART_INF_F) ? exp2f(t2[n] - lse2) : 0.f;
          ds[n] = pr * (dp[n] - dl);
        }
        store_row32<BK>(sS, tid, c32 * 32, ds, st.lam);
      }
    }
    tc_fence_before();
    if (MODE == 1) {
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t as = smem_u32(sS), bk = smem_u32(sK);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_f16(tAcc, sdesc_sw128(as + (k / 4) * (128 * 128) + (k % 4) * 32, 16, 1024),
                  sdesc_sw128(bk + k * 2048, BK * 128, 1024), ID_DQ, (first && k == 0) ? 0u : 1u);
        mma_commit(&bars[1]);
      }
      if (!mbar_wait_bounded(&bars[1], mma_phase, kWaitLimitNs)) {
        *s_abort = 1;
        record_error(p.err, kErrTimeout);
      }
      mma_phase ^= 1;
      tc_fence_after();
      first = false;
    }
    __syncthreads();
    if (*s_abort) break;
  }

  // epilogue
  if (MODE == 0) {
    if (rvalid) {
      float* o = p.part + (((size_t)split * p.Hkv + hk) * R + r) * 3;
      o[0] = m2, o[1] = l, o[2] = sd;
    }
  } else {
    // every lane takes part in the warp-wide TMEM loads; only valid rows store
    float* out = !rvalid ? nullptr
                 : p.nsplit == 1 ? p.dQ + ((size_t)i * p.H + h) * D
                                 : p.dqpart + (((size_t)split * p.Hkv + hk) * R + r) * D;
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
      float v[32];
      if (!first) {
        tmem_ld32(tAcc + lane_off + c, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
      if (out) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(out + c + e) =
              make_float4(v[e] * st.dq_fac, v[e + 1] * st.dq_fac, v[e + 2] * st.dq_fac, v[e + 3] * st.dq_fac);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// Merge the split partials: lse and delta outputs plus the gradient passes' per-row values.
__global__ void __launch_bounds__(256) k_lse_merge(Params p) {
  const long idx = (long)blockIdx.x * 256 + threadIdx.x;
  if (idx >= (long)p.Hkv * p.R) return;
  const int hk = (int)(idx / p.R), r = (int)(idx % p.R);
  float m2 = -CUDART_INF_F;
  for (int s = 0; s < p.nsplit; ++s) m2 = fmaxf(m2, p.part[(((size_t)s * p.Hkv + hk) * p.R + r) * 3]);
  float l = 0.f, sd = 0.f;
  if (m2 > -CUDART_INF_F) {
    for (int s = 0; s < p.nsplit; ++s) {
      const float* q = p.part + (((size_t)s * p.Hkv + hk) * p.R + r) * 3;
      if (q[0] == -CUDART_INF_F) continue;
      const float f = exp2f(q[0] - m2);
      l = fmaf(q[1], f, l);
      sd = fmaf(q[2], f, sd);
    }
  }
  const int i = r / p.G, h = hk * p.G + r % p.G;
  const Stats* st = p.st;
  if (l > 0.f) {
    const float lse2 = m2 + log2f(l);
    const float dl = sd / l;
    p.lse2[idx] = lse2;
    p.dlt[idx] = dl;
    p.lse[(size_t)i * p.H + h] = lse2 * kLn2;
    p.delta[(size_t)i * p.H + h] = dl * st->delta_fac + p.dOr[idx];
  } else {
    p.lse2[idx] = -CUDART_INF_F;
    p.dlt[idx] = 0.f;
    p.lse[(size_t)i * p.H + h] = -CUDART_INF_F;
    p.delta[(size_t)i * p.H + h] = 0.f;
  }
}

// dQ = sum of the split partials, in split order.
__global__ void __launch_bounds__(256) k_dq_reduce(Params p) {
  const long nv = (long)p.Hkv * p.R * (p.D / 4);
  const long idx = (long)blockIdx.x * 256 + threadIdx.x;
  if (idx >= nv) return;
  const long row = idx / (p.D / 4);
  const int c = (int)(idx % (p.D / 4)) * 4;
  const int hk = (int)(row / p.R), r = (int)(row % p.R);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < p.nsplit; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(p.dqpart + (((size_t)s * p.Hkv + hk) * p.R + r) * p.D + c);
    acc.x += x.x, acc.y += x.y, acc.z += x.z, acc.w += x.w;
  }
  const int i = r / p.G, h = hk * p.G + r % p.G;
  *reinterpret_cast<float4*>(p.dQ + ((size_t)i * p.H + h) * p.D + c) = acc;
}

// ------------------------------------------------------------------------------------------------
// key-tile pass: dK and dV

template <int D, int Dv, int BK>
struct ColsCfg {
  static constexpr int KB = BK * D * 2, VB = BK * Dv * 2, QB = 128 * D * 2, OB = 128 * Dv * 2, PB = 128 * BK * 2;
  static constexpr int OFF_K = 0, OFF_V = KB, OFF_Q = KB + VB, OFF_O = OFF_Q + QB, OFF_P = OFF_O + OB,
                       OFF_S = OFF_P + PB, OFF_BAR = OFF_S + PB;
  static constexpr int SMEM = OFF_BAR + 64 + 1024;
  static constexpr int NDH = D >= 128 ? D / 128 : 1, NVH = Dv >= 128 ? Dv / 128 : 1;
  static constexpr int TCOLS = pow2_at_least(2 * BK + (NDH + NVH) * BK);
};

template <int D, int Dv, int BK>
__global__ void __launch_bounds__(128, 1)
    k_cols(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO, Params p) {
  using C = ColsCfg<D, Dv, BK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sO = sm + C::OFF_O;
  uint8_t* sP = sm + C::OFF_P;
  uint8_t* sS = sm + C::OFF_S;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 16);
  int* s_abort = reinterpret_cast<int*>(sm + C::OFF_BAR + 20);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int kt = blockIdx.x, hk = blockIdx.y;
  const int j0 = kt * BK;
  const int R = p.R, G = p.G;

  // first row tile that can see key j0 under the causal tail
  int qt_begin = 0;
  if (p.causal) {
    const long imin = (long)j0 - ((long)p.M - p.N);
    if (imin > 0) qt_begin = (int)min((long)p.nQT, (imin * G) / 128);
  }
  bool have = qt_begin < p.nQT && R > 0;

  if (warp == 0) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    *s_abort = 0;
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase, tP = tbase + BK, tV = tbase + 2 * BK, tK = tbase + 2 * BK + C::NVH * BK;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const Stats st = *p.st;

  if (have) {
    decode_tile<D, BK, 128>(p.k, p.k_type, p.rbk, hk, p.Hkv, j0, p.M, sK, st.sK, nullptr);
    decode_tile<Dv, BK, 128>(p.v, p.v_type, p.rbv, hk, p.Hkv, j0, p.M, sV, st.sV, p.rmean + (size_t)hk * Dv);
    fence_proxy_async_smem();
  }
  __syncthreads();

  constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
  constexpr uint32_t ID_T = idesc_f16(128, BK, true, true);
  constexpr uint32_t LBO_O = Dv >= 128 ? 128 * 128 : 0;  // second 64-row block of dO^T (duplicate if Dv = 64)
  constexpr uint32_t LBO_Q = D >= 128 ? 128 * 128 : 0;
  uint32_t tma_phase = 0, mma_phase = 0;
  bool first = true;

  for (int qt = qt_begin; have && qt < p.nQT; ++qt) {
    const int r0 = qt * 128;
    if (tid == 0) {
      mbar_arrive_expect_tx(&bars[0], (uint32_t)(C::QB + C::OB));
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * 128 * 128, &tmQ, &bars[0], c * 64, r0, hk);
#pragma unroll
      for (int c = 0; c < Dv / 64; ++c) tma_load_3d(sO + c * 128 * 128, &tmO, &bars[0], c * 64, r0, hk);
    }
    const int r = r0 + tid;
    const bool rvalid = r < R;
    const int i = rvalid ? r / G : 0;
    const int h = hk * G + (rvalid ? r % G : 0);
    const float lse2 = rvalid ? p.lse2[(size_t)hk * R + r] : -CUDART_INF_F;
    const float dl = rvalid ? p.dlt[(size_t)hk * R + r] : 0.f;
    const bool live = lse2 > -CUDART_INF_F;
    const long jlast = rvalid ? (p.causal ? min((long)p.M - 1, (long)p.M - p.N + i) : (long)p.M - 1) : -1;
    const uint16_t* mrow = p.mask ? p.mask + ((size_t)(h % p.Hm) * p.N + i) * p.M : nullptr;

    if (!mbar_wait_bounded(&bars[0], tma_phase, kWaitLimitNs)) {
      *s_abort = 1;
      record_error(p.err, kErrTimeout);
    }
    tma_phase ^= 1;
    __syncthreads();
    if (*s_abort) break;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t aq = smem_u32(sQ), ao = smem_u32(sO), bk = smem_u32(sK), bv = smem_u32(sV);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_f16(tS, sdesc_sw128(aq + (k / 4) * (128 * 128) + (k % 4) * 32, 16, 1024),
                sdesc_sw128(bk + (k / 4) * (BK * 128) + (k % 4) * 32, 16, 1024), ID_S, k > 0);
#pragma unroll
      for (int k = 0; k < Dv / 16; ++k)
        mma_f16(tP, sdesc_sw128(ao + (k / 4) * (128 * 128) + (k % 4) * 32, 16, 1024),
                sdesc_sw128(bv + (k / 4) * (BK * 128) + (k % 4) * 32, 16, 1024), ID_S, k > 0);
      mma_commit(&bars[1]);
    }
    if (!mbar_wait_bounded(&bars[1], mma_phase, kWaitLimitNs)) {
      *s_abort = 1;
      record_error(p.err, kErrTimeout);
    }
    mma_phase ^= 1;
    tc_fence_after();

#pragma unroll 1
    for (int c32 = 0; c32 < BK / 32; ++c32) {
      float s[32], dp[32];
      tmem_ld32(tS + lane_off + c32 * 32, s);
      tmem_ld32(tP + lane_off + c32 * 32, dp);
      tmem_ld_wait();
      const int jb = j0 + c32 * 32;
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        const int j = jb + n;
        bool ok = live && (long)j <= jlast;
        float mv = 0.f;
        if (ok && mrow) {
          mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
          ok = !(mv == -CUDART_INF_F);
        }
        const float pr = ok ? exp2f(fmaf(s[n], st.c2, mv * kLog2e) - lse2) : 0.f;
        s[n] = pr;
        dp[n] = pr * (dp[n] - dl);
      }
      store_row32<BK>(sP, tid, c32 * 32, s, st.sP);
      store_row32<BK>(sS, tid, c32 * 32, dp, st.lam);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ao = smem_u32(sO), aq = smem_u32(sQ), bp = smem_u32(sP), bs = smem_u32(sS);
#pragma unroll
      for (int hh = 0; hh < C::NVH; ++hh)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16(tV + hh * BK, sdesc_sw128(ao + hh * 2 * (128 * 128) + k * 2048, LBO_O, 1024),
                  sdesc_sw128(bp + k * 2048, 128 * 128, 1024), ID_T, (first && k == 0) ? 0u : 1u);
#pragma unroll
      for (int hh = 0; hh < C::NDH; ++hh)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16(tK + hh * BK, sdesc_sw128(aq + hh * 2 * (128 * 128) + k * 2048, LBO_Q, 1024),
                  sdesc_sw128(bs + k * 2048, 128 * 128, 1024), ID_T, (first && k == 0) ? 0u : 1u);
      mma_commit(&bars[1]);
    }
    if (!mbar_wait_bounded(&bars[1], mma_phase, kWaitLimitNs)) {
      *s_abort = 1;
      record_error(p.err, kErrTimeout);
    }
    mma_phase ^= 1;
    tc_fence_after();
    first = false;
    __syncthreads();
    if (*s_abort) break;
  }

  // epilogue: lane = feature row (dv or d), columns = keys
  {
    const int lrow = warp * 32 + (tid & 31);
#pragma unroll 1
    for (int hh = 0; hh < C::NVH; ++hh) {
      const int dv = hh * 128 + lrow;
#pragma unroll 1
      for (int c = 0; c < BK; c += 32) {
        float v[32];
        if (!first) {
          tmem_ld32(tV + hh * BK + lane_off + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (dv < Dv) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = j0 + c + e;
            if (j < p.M) p.dV[((size_t)j * p.Hkv + hk) * Dv + dv] = v[e] * st.dv_fac;
          }
        }
      }
    }
#pragma unroll 1
    for (int hh = 0; hh < C::NDH; ++hh) {
      const int d = hh * 128 + lrow;
#pragma unroll 1
      for (int c = 0; c < BK; c += 32) {
        float v[32];
        if (!first) {
          tmem_ld32(tK + hh * BK + lane_off + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (d < D) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = j0 + c + e;
            if (j < p.M) p.dK[((size_t)j * p.Hkv + hk) * D + d] = v[e] * st.dk_fac;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// Fill kernel for degenerate shapes (a value into n floats).
__global__ void k_fill(float* x, long n, float v) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < n) x[idx] = v;
}

}  // namespace fab
