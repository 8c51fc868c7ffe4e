// Device code of the flash-attention backward over a raw K/V cache (sm_103a).
//
// Pipeline (all on one stream, see fa_back.cu; the plan level depends on the workspace):
//   k_row_stats  -> per-block max |x| and max row norm of Q, dO, K^ and V^
//   k_vsum       -> per-chunk column sums of V^ (for its column mean r)
//   k_finalize   -> power-of-two operand scales, r, the dS multiplier
//   k_convert    -> Q, dO as scaled binary16 rows packed per KV head (row r = i*G + g)
//   k_predecode  -> binary16 K', V' copies of the cache (levels 2 and 1)
//   k_rows3/k_rows2 <LSE> -> per (row tile, key split): running max / sum / sum of p*dP
//                            (TMA-fed from the copies, or decoding raw rows in the CTA at level 0)
//   k_lse_merge  -> lse, delta outputs; log2-domain lse and shifted delta for the gradient passes
//   k_cols2      -> dK^T = scale * Q^T dS and dV^T = dO^T P per key tile; stores dS (level 2)
//   k_dq_gemm    -> dQ = scale * dS K' per row tile over the stored dS (level 2), or
//   k_rows3/k_rows2 <DQ> -> dQ recomputing S, dP, dS per row tile (levels 1, 0);
//                           both split over keys and merged in fixed order (k_dq_reduce)
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
#include <climits>
#include <stdint.h>

#include "sm100.cuh"

namespace fab {

constexpr int kTypeF32 = 0, kTypeF16 = 1, kTypeQ8 = 2, kTypeQ4 = 3;
constexpr int kErrTimeout = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait (and per drain after an abort)
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
  int lamr_exp;  // largest exponent of the per-row dS multipliers (raised by k_convert)
  // score extensions (ext_scores): the soft cap's argument u = cu * (Q.K accumulator) =
  // scale q.k / c and its height c log2(e); both 0 without a cap
  float cu, cap2;
};

// The dS stored for the dQ product takes each row's own multiplier only when some row's exceeds
// the common one by more than 2^12.  A row within that gap has its largest |dS| value no more
// than 2^12 below the common scale's 2^15, so its values stay far inside binary16's normal range
// and keep its relative precision; the per-row copy costs the dK/dV pass extra shared-memory
// traffic, so typical inputs (rows of similar size) skip it.
constexpr int kRowScaleGap = 12;
__device__ __forceinline__ bool rows_need_own_scale(const Stats& st) {
  return st.lamr_exp - ilogbf(st.lam) > kRowScaleGap;
}

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
  float* rsh;     // [Hkv][Dv]  -r' * sV, an exact binary16 value (the decoders' V shift)
  __half* kd;     // [Hkv][D/64][M][64]   binary16 K' = k^ sK, panel-major (TMA-fed passes; else null)
  __half* vd;     // [Hkv][Dv/64][M][64]  binary16 V' = v^ sV - r' sV
  float* o_out;   // [N][H][Dv] forward output O (fa_forward), or null
  float* lamr;    // [Hkv][R]  per-row multiplier of dS for the dQ product (power of two), from
                  //           the row's own |dO_i| bound, so small rows keep binary16 precision
  __half* ds;     // binary16 lamr * dS from the dK/dV pass, read by k_dq_gemm (or null): contiguous
                  // [128 rows][64 keys] tiles, tile (hk, row tile qt, key tile kt64) at
                  // (hk * nQT + qt) * ldds + kt64
  int ldds;       // 64-key tiles per row tile (whole gradient-pass key tiles)
  const float* lse_in;    // [N][H] given row lse (natural log; fa_back_with_stats), or null
  const float* delta_in;  // [N][H] given row delta = rowsum(dO o O), or null
  // raw K/V staging of the row passes
  int raw_bulk;        // 1: rows are 16-byte multiples, copied by bulk async copies; 0: 4-byte async copies
  int rbk_pad, rbv_pad;  // raw row strides in shared memory (16-byte multiples)
  int ke;              // keys per raw ring entry
  int raw_depth;       // entries of the K ring (2..8)
  int raw_depth_v;     // entries of the V ring (1..8)
  int* err;
  uint64_t wait_ns;    // a wait gives up after this long: kWaitLimitNs, shorter only under the
                       // failure-detection hook (fa_back_test_wait_limit); drains keep kWaitLimitNs
  // score extensions (fa_back_ext); all null / 0 for the plain operation
  float softcap;       // c > 0: the score x = scale q.k becomes c tanh(x / c); 0: none
  const float* alibi;  // [H] slopes: bias slope_h (j - (M - N + i)) added after the mask, or null
  const float* sinks;  // [H] sink logits joining every row's softmax denominator, or null
  float* dsinks;       // [H] gradient of the sink logits (with sinks), or null
  float* sg;           // [Hkv][R] per-row sink-gradient terms, summed per head by k_sink_grad
};

__host__ __device__ constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

// ------------------------------------------------------------------------------------------------
// decoding raw cache rows

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Byte offset of the 8-value unit (row, c0) in a tile of DD/64 panels of [rows][64] binary16
// (128-byte rows, 128-byte swizzle).
__device__ __forceinline__ uint32_t panel_off_u(int rows, int row, int c0) {
  return (uint32_t)(c0 >> 6) * (uint32_t)(rows * 128) + swz128((uint32_t)row * 128 + (uint32_t)((c0 & 63) >> 3) * 16);
}

// Two 8-bit values b0, b1 (bits 0..15 of x, already biased to 0..255) as binary16 1024 + b:
// the bytes are placed under the exponent byte 0x64, which makes the mantissa the value.
__device__ __forceinline__ __half2 bytes_as_h2_plus1024(uint32_t x) {
  return u32_as_h2(__byte_perm(x, 0x64646464u, 0x5140));
}

// The shifts of columns c0..c0+7 (c0 % 8 == 0) as binary16 pairs; zeros where shift is null.
__device__ __forceinline__ void shift8_h(const float* shift, int c0, __half2* sh) {
  if (shift) {  // two aligned 16-byte loads
    const float4 a = *reinterpret_cast<const float4*>(shift + c0), b = *reinterpret_cast<const float4*>(shift + c0 + 4);
    sh[0] = __floats2half2_rn(a.x, a.y), sh[1] = __floats2half2_rn(a.z, a.w);
    sh[2] = __floats2half2_rn(b.x, b.y), sh[3] = __floats2half2_rn(b.z, b.w);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) sh[e] = __floats2half2_rn(0.f, 0.f);
  }
}

// Decode 8 consecutive values c0..c0+7 (c0 % 8 == 0) of a raw row into four packed binary16
// pairs, out = x^ * sig - shift (sh: the shifts from shift8_h, each an exact binary16 value).
// Codes are turned into exact binary16 integers in pairs; one fused multiply-add then applies
// the block scale, the power-of-two operand scale and the shift with a single rounding.  The
// row pointer may point to global or shared memory.
__device__ __forceinline__ uint4 decode8_h_sh(const uint8_t* row, int type, int c0, float sig, const __half2* sh) {
  uint32_t w[4];
  if (type == kTypeQ8 || type == kTypeQ4) {
    const bool q8 = type == kTypeQ8;
    const uint8_t* b = row + (q8 ? 34 : 18) * (c0 >> 5);
    const float d = __half2float(*reinterpret_cast<const __half*>(b));
    const __half2 ds = __float2half2_rn(d * sig);
    const int o = c0 & 31;
    const uint16_t* cp = reinterpret_cast<const uint16_t*>(b + 2 + (q8 ? o : (o & 15)));
    const __half2 bias = q8 ? __float2half2_rn(1152.f) : __float2half2_rn(1032.f);
    const int sh4 = (o >= 16) ? 4 : 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t pr = cp[e];
      const uint32_t x = q8 ? (pr ^ 0x8080u) : ((pr >> sh4) & 0x0f0fu);
      const __half2 code = __hsub2(bytes_as_h2_plus1024(x), bias);  // q8_0: int8 code; q4_0: nibble - 8
      w[e] = h2_as_u32(__hfma2(code, ds, sh[e]));
    }
  } else if (type == kTypeF16) {
    // in f32: the power-of-two scale can exceed binary16's range (small-magnitude caches);
    // x * sig is exact there, so the one rounding is the final conversion
    const uint4 u = *reinterpret_cast<const uint4*>(row + 2 * c0);
    const uint32_t in[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __half22float2(u32_as_h2(in[e])), f = __half22float2(sh[e]);
      w[e] = h2_as_u32(__floats2half2_rn(fmaf(x.x, sig, f.x), fmaf(x.y, sig, f.y)));
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(row + 4 * c0);
    const float4 c = *reinterpret_cast<const float4*>(row + 4 * c0 + 16);
    const float x[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(sh[e]);
      w[e] = h2_as_u32(__floats2half2_rn(fmaf(x[2 * e], sig, f.x), fmaf(x[2 * e + 1], sig, f.y)));
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 decode8_h(const uint8_t* row, int type, int c0, float sig, const float* shift) {
  __half2 sh[4];
  shift8_h(shift, c0, sh);
  return decode8_h_sh(row, type, c0, sig, sh);
}

// ---- decoders of the row passes: raw rows staged in shared memory -> binary16 operand tiles
//
// A decoder thread owns one column group of every row it handles: a whole 32-value block for
// q8_0 / q4_0 (one scale load, the codes read as aligned 32-bit words), 8 values for f16 / f32.
// Its V shifts are therefore fixed and held in registers.
__device__ __forceinline__ int group_cols(int type) { return (type == kTypeQ8 || type == kTypeQ4) ? 32 : 8; }

// Decoder thread -> (group, first row, row step).  For q8_0/q4_0 the 8 lanes of a quarter-warp
// take one column group of 8 consecutive rows, so their 16-byte stores hit 8 distinct bank
// groups of the swizzled tile; for f16/f32 they take 8 consecutive groups of one row.
// With 8 blocks per row (D = 256) a warp's four groups are chosen so that their codes start at
// word offsets of distinct residues mod 4 in the raw row: raw rows are 68 (q8_0) or 36 (q4_0)
// words apart, so 8 rows x 4 groups then cover all 32 banks and the raw loads are
// conflict-free (groups {0,1,3,5} and {7,2,4,6}).
__device__ __forceinline__ void decoder_map(int type, int DD, int NT, int dt, int& g, int& r0, int& rs) {
  const int ng = DD / group_cols(type);
  if (type == kTypeQ8 || type == kTypeQ4) {
    const int gs = (dt >> 3) % ng;
    g = ng == 8 ? (int)((0x64275310u >> (4 * gs)) & 7u) : gs;
    r0 = (dt & 7) + 8 * (dt / (8 * ng));
  } else {
    g = dt % ng;
    r0 = dt / ng;
  }
  rs = NT / ng;
}

template <int DD, int NT>
__device__ __forceinline__ void load_group_shift(const float* shift, int type, int dt, __half2* sh) {
  int g, r0, rs;
  decoder_map(type, DD, NT, dt, g, r0, rs);
  const int cg = group_cols(type);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int c = g * cg + 2 * e;
    sh[e] = (2 * e < cg) ? __floats2half2_rn(shift[c], shift[c + 1]) : __float2half2_rn(0.f);
  }
}

// Decode raw rows 0..nrows-1 of one staged entry (shared address raw0, stride rb_pad) into
// rows prow0.. of a tile of DD/64 panels of [BKR][64]; rows >= nvalid become zero.
//
// q8_0 / q4_0: the codes of a block start 2 bytes in, so they are 4-byte aligned for every
// other block; either way each pair of codes sits inside one aligned 32-bit word (aligned codes:
// bytes (0,1) and (2,3) of word k; otherwise bytes (2,3) of word k and (0,1) of word k+1).  One
// byte permute per pair puts the two biased codes under the binary16 exponent byte 0x64 (value
// 1024 + byte), one subtraction removes the bias exactly, and one fused multiply-add applies
// d * sigma and the shift with a single rounding.
template <int DD, int BKR, int NT, bool SHIFT>
__device__ __forceinline__ void decode_rows(int type, uint32_t raw0, int rb_pad, int nrows, int nvalid, int prow0,
                                            uint32_t panels, float sig, const __half2* sh, int dt) {
  int g, rfirst, rs;
  decoder_map(type, DD, NT, dt, g, rfirst, rs);
  const __half2 z = __float2half2_rn(0.f);
  if (type == kTypeQ8 || type == kTypeQ4) {
    const bool q8 = type == kTypeQ8;
    const int bbytes = q8 ? 34 : 18;
    const __half2 bias = q8 ? __float2half2_rn(1152.f) : __float2half2_rn(1032.f);
    for (int rr = rfirst; rr < nrows; rr += rs) {
      uint32_t o[16];
      if (rr < nvalid) {
        const uint32_t blk = raw0 + rr * rb_pad + g * bbytes;
        // d * sigma in f32 (sigma may exceed binary16's range), rounded once to binary16
        const __half2 ds = __float2half2_rn(h2f((uint16_t)lds_u16(blk)) * sig);
        const uint32_t cs = blk + 2, cb = cs & ~3u;
        const bool al = (cs & 3u) == 0;
        const uint32_t sa = al ? 0x5140u : 0x7362u, sb = al ? 0x7362u : 0x5140u;
        if (q8) {
          uint32_t w[9];
#pragma unroll
          for (int k = 0; k < 9; ++k) w[k] = lds_u32(cb + 4 * k) ^ 0x80808080u;  // codes + 128
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t wa = w[k], wb = al ? w[k] : w[k + 1];
            const __half2 c0 = __hsub2(u32_as_h2(__byte_perm(wa, 0x64646464u, sa)), bias);
            const __half2 c1 = __hsub2(u32_as_h2(__byte_perm(wb, 0x64646464u, sb)), bias);
            o[2 * k] = h2_as_u32(__hfma2(c0, ds, SHIFT ? sh[2 * k] : z));
            o[2 * k + 1] = h2_as_u32(__hfma2(c1, ds, SHIFT ? sh[2 * k + 1] : z));
          }
        } else {
          uint32_t w[5];
#pragma unroll
          for (int k = 0; k < 5; ++k) w[k] = lds_u32(cb + 4 * k);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t wa = w[k], wb = al ? w[k] : w[k + 1];
            const uint32_t la = wa & 0x0f0f0f0fu, lb = wb & 0x0f0f0f0fu;                // values 4k.. (low nibbles)
            const uint32_t ha = (wa >> 4) & 0x0f0f0f0fu, hb = (wb >> 4) & 0x0f0f0f0fu;  // values 16+4k.. (high)
            const __half2 c0 = __hsub2(u32_as_h2(__byte_perm(la, 0x64646464u, sa)), bias);
            const __half2 c1 = __hsub2(u32_as_h2(__byte_perm(lb, 0x64646464u, sb)), bias);
            const __half2 c2 = __hsub2(u32_as_h2(__byte_perm(ha, 0x64646464u, sa)), bias);
            const __half2 c3 = __hsub2(u32_as_h2(__byte_perm(hb, 0x64646464u, sb)), bias);
            o[2 * k] = h2_as_u32(__hfma2(c0, ds, SHIFT ? sh[2 * k] : z));
            o[2 * k + 1] = h2_as_u32(__hfma2(c1, ds, SHIFT ? sh[2 * k + 1] : z));
            o[8 + 2 * k] = h2_as_u32(__hfma2(c2, ds, SHIFT ? sh[8 + 2 * k] : z));
            o[8 + 2 * k + 1] = h2_as_u32(__hfma2(c3, ds, SHIFT ? sh[8 + 2 * k + 1] : z));
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) o[k] = 0u;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
        sts_v4(panels + panel_off_u(BKR, prow0 + rr, g * 32 + 8 * m), o[4 * m], o[4 * m + 1], o[4 * m + 2],
               o[4 * m + 3]);
    }
  } else {
    const bool f16 = type == kTypeF16;
    for (int rr = rfirst; rr < nrows; rr += rs) {
      uint32_t o[4] = {0u, 0u, 0u, 0u};
      if (rr < nvalid) {
        const uint32_t a = raw0 + rr * rb_pad + g * (f16 ? 16 : 32);
        if (f16) {
          const uint4 v = lds_v4(a);
          const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // in f32, as decode8_h
            const float2 x = __half22float2(u32_as_h2(in[e])), f = __half22float2(SHIFT ? sh[e] : z);
            o[e] = h2_as_u32(__floats2half2_rn(fmaf(x.x, sig, f.x), fmaf(x.y, sig, f.y)));
          }
        } else {
          const uint4 u0 = lds_v4(a), u1 = lds_v4(a + 16);
          const uint32_t in[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(SHIFT ? sh[e] : z);
            o[e] = h2_as_u32(__floats2half2_rn(fmaf(__uint_as_float(in[2 * e]), sig, f.x),
                                               fmaf(__uint_as_float(in[2 * e + 1]), sig, f.y)));
          }
        }
      }
      sts_v4(panels + panel_off_u(BKR, prow0 + rr, g * 8), o[0], o[1], o[2], o[3]);
    }
  }
}

// Byte offset of 8-value unit (row, c0) in a tile of DD/64 panels of [rows][64] binary16.
__device__ __forceinline__ uint32_t panel_off(int rows, int row, int c0) {
  return (uint32_t)(c0 >> 6) * (uint32_t)(rows * 128) + swz128((uint32_t)row * 128 + (uint32_t)((c0 & 63) >> 3) * 16);
}

// Decode BK cache rows (keys j0.., KV head hk) straight from global memory into a binary16
// operand tile (DD/64 panels of [BK rows][64 columns], 128-byte swizzled).  Keys >= M become zero.
template <int DD, int BK, int NT>
__device__ __forceinline__ void decode_tile(const uint8_t* base, int type, int rb, int hk, int Hkv, int j0, int M,
                                            uint8_t* panels, float sigma, const float* shift, int tid) {
  constexpr int UPR = DD / 8;
  const uint32_t pu = smem_u32(panels);
  for (int u = tid; u < BK * UPR; u += NT) {
    const int row = u / UPR;
    const int c0 = (u % UPR) * 8;
    const int j = j0 + row;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (j < M) w = decode8_h(base + ((size_t)j * Hkv + hk) * rb, type, c0, sigma, shift);
    sts_v4(pu + panel_off(BK, row, c0), w);
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

// ---- score extensions: soft cap, ALiBi bias (and, in k_lse_merge, sink logits)
//
// Log2-domain exponents of one 32-key chunk (keys j0 .. j0+31, row r of KV head hk) with the
// extensions applied in this order: x = scale q.k (the Q.K accumulator s[n] times c2), the soft
// cap c tanh(x / c) (when st.cap2 > 0), the mask, the ALiBi bias slope_h (j - (M - N + i)), and
// the row offset t2off.  Masked keys get -inf.  tanh(u) = sign(u) (1 - 2w) with w = 1 / (1 +
// e^{2|u|}) (the exponential form of tanh), whose derivative is 1 - tanh^2 = 4 w (1 - w); computed
// this way the derivative keeps its relative precision where tanh is close to one.
//   FAC 0: exponents only (LSE/D passes);
//   FAC 1: log2 of the derivative added to the exponent (dQ passes: the exponential is then
//          lam p (1 - tanh^2), the multiplier of (dP - delta) in dS);
//   FAC 2: dp[n] replaced by (dp[n] - dl)(1 - tanh^2) (the dK/dV pass, which needs p itself for
//          dV; it then subtracts 0 instead of dl).
// Only the passes' EXT variants contain it; the plain operation's kernels are built without.
template <int FAC>
__device__ __forceinline__ void ext_scores(float* s, float* dp, int j0, int r, int hk, float t2off, float dl,
                                           long jlast, const uint16_t* mrow, const Stats& st, const float* slopes,
                                           int G, int diag0) {
  const int i = r / G, h = hk * G + r % G;
  const float sl2 = slopes ? __ldg(slopes + h) * kLog2e : 0.f;
  const long jd = (long)diag0 + i;  // the query's position on the key axis
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    const int j = j0 + n;
    bool ok = (long)j <= jlast;
    float mv = 0.f;
    if (ok && mrow) {
      mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
      ok = !(mv == -CUDART_INF_F);
    }
    float y, f = 1.f;
    if (st.cap2 > 0.f) {
      const float u = s[n] * st.cu;
      const float w = __frcp_rn(1.f + ex2(fabsf(u) * (2.f * kLog2e)));
      y = st.cap2 * copysignf(1.f - 2.f * w, u);
      f = 4.f * w * (1.f - w);
    } else {
      y = s[n] * st.c2;
    }
    float t = ok ? y + fmaf(mv, kLog2e, fmaf(sl2, (float)((long)j - jd), t2off)) : -CUDART_INF_F;
    if (FAC == 1) t += __log2f(f);  // f = 0 (a saturated cap) gives -inf: no contribution
    s[n] = t;
    if (FAC == 2) dp[n] = ok ? (dp[n] - dl) * f : 0.f;
  }
}

// ------------------------------------------------------------------------------------------------
// statistics and packing

// Values c0 .. c0+7 of a raw cache row, decoded exactly to f32 (code * d, or the stored value).
// MAGIC selects how an 8-bit code becomes a float (both exact): an int-to-float conversion, or the
// byte placed under a float's exponent (fewer conversions, more registers)
template <bool MAGIC = false>
__device__ __forceinline__ void decode8_f(const uint8_t* row, int type, int c0, float* x) {
  if ((type == kTypeQ8 || type == kTypeQ4) && !MAGIC) {
    const bool q8 = type == kTypeQ8;
    const uint8_t* b = row + (q8 ? 34 : 18) * (c0 >> 5);
    const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
    const int o = c0 & 31;
    const uint16_t* cp = reinterpret_cast<const uint16_t*>(b + 2 + (q8 ? o : (o & 15)));
    const int sh = o >= 16 ? 4 : 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t pr = __ldg(cp + e);
      if (q8) {
        x[2 * e] = (float)(int8_t)(pr & 0xffu) * d;
        x[2 * e + 1] = (float)(int8_t)(pr >> 8) * d;
      } else {
        x[2 * e] = (float)((int)((pr >> sh) & 15u) - 8) * d;
        x[2 * e + 1] = (float)((int)((pr >> (8 + sh)) & 15u) - 8) * d;
      }
    }
  } else if (type == kTypeQ8 || type == kTypeQ4) {
    const bool q8 = type == kTypeQ8;
    const uint8_t* b = row + (q8 ? 34 : 18) * (c0 >> 5);
    const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
    const int o = c0 & 31;
    const uint16_t* cp = reinterpret_cast<const uint16_t*>(b + 2 + (q8 ? o : (o & 15)));
    const int sh = (!q8 && o >= 16) ? 4 : 0;
    // each code as a biased byte under the exponent of 1.5 * 2^23, which makes the byte the low
    // mantissa bits: subtracting 1.5 * 2^23 plus the bias gives the code exactly (no int-to-float
    // conversion), and code * d is exact in f32
    const float off = q8 ? 12583040.f : 12582920.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t w = (uint32_t)__ldg(cp + 2 * e) | ((uint32_t)__ldg(cp + 2 * e + 1) << 16);
      const uint32_t bb = q8 ? (w ^ 0x80808080u) : ((w >> sh) & 0x0f0f0f0fu);
#pragma unroll
      for (int k = 0; k < 4; ++k) x[4 * e + k] = (__uint_as_float(__byte_perm(bb, 0x4B400000u, 0x7650 | k)) - off) * d;
    }
  } else if (type == kTypeF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + 2 * c0));
    const uint32_t in[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(u32_as_h2(in[e]));
      x[2 * e] = f.x, x[2 * e + 1] = f.y;
    }
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(row + 4 * c0));
    const float4 c = __ldg(reinterpret_cast<const float4*>(row + 4 * c0 + 16));
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = c.x, x[5] = c.y, x[6] = c.z, x[7] = c.w;
  }
}

// max |x| and the sum of x^2 over values c0 .. c0+7 of a row.  For q8_0 and q4_0 both come from
// the codes by four-way byte arithmetic: max |code| times |d| (exact, as the decoded values'
// maximum is) and the integer sum of code^2 times d^2.
template <int TYPE>
__device__ __forceinline__ void values8_stats(const uint8_t* row, int c0, float& am, float& ss) {
  if constexpr (TYPE == kTypeQ8 || TYPE == kTypeQ4) {
    constexpr bool q8 = TYPE == kTypeQ8;
    const uint8_t* b = row + (q8 ? 34 : 18) * (c0 >> 5);
    const float d = h2f(__ldg(reinterpret_cast<const unsigned short*>(b)));
    const int o = c0 & 31;
    const uint16_t* cp = reinterpret_cast<const uint16_t*>(b + 2 + (q8 ? o : (o & 15)));
    uint32_t w[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      w[e] = (uint32_t)__ldg(cp + 2 * e) | ((uint32_t)__ldg(cp + 2 * e + 1) << 16);
      if (!q8) w[e] = __vsub4((w[e] >> (o >= 16 ? 4 : 0)) & 0x0f0f0f0fu, 0x08080808u);  // signed codes
    }
    // per-byte |code|, read as unsigned (the code -128 gives the byte 0x80, i.e. 128)
    const uint32_t a = __vmaxu4(__vabs4(w[0]), __vabs4(w[1]));
    const uint32_t m = max(max(a & 0xffu, (a >> 8) & 0xffu), max((a >> 16) & 0xffu, a >> 24));
    const int q2 = __dp4a((int)w[0], (int)w[0], __dp4a((int)w[1], (int)w[1], 0));
    am = (float)m * fabsf(d);
    ss = (float)q2 * (d * d);
  } else {
    float x[8];
    decode8_f(row, TYPE, c0, x);
    am = 0.f, ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(x[e])), ss = fmaf(x[e], x[e], ss);
  }
}

// Sums over the 32 lanes of four values at once (six exchanges instead of twenty): lane l ends
// with the sum of value 2 * bit4(l) + bit3(l).
__device__ __forceinline__ float warp_sum4(const float* a, int lane) {
  const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
  const float b0 = (h16 ? a[2] : a[0]) + __shfl_xor_sync(0xffffffffu, h16 ? a[0] : a[2], 16);
  const float b1 = (h16 ? a[3] : a[1]) + __shfl_xor_sync(0xffffffffu, h16 ? a[1] : a[3], 16);
  float c = (h8 ? b1 : b0) + __shfl_xor_sync(0xffffffffu, h8 ? b0 : b1, 8);
  c += __shfl_xor_sync(0xffffffffu, c, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// One tensor's rows (nrows rows of DD values, rstride bytes apart), one warp per row and four rows
// per step (lane = 8 consecutive values): this lane's max |x| and max squared row norm.
template <int TYPE>
__device__ __forceinline__ void rows_stats(const uint8_t* base, long nrows, size_t rstride, int DD, long gw,
                                           long nw, int lane, float& amx, float& nrm) {
  const int c0 = lane * 8;
  const bool on = c0 < DD;
  for (long r0 = gw; r0 < nrows; r0 += 4 * nw) {
    float am[4], ss[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long r = r0 + u * nw;
      am[u] = 0.f, ss[u] = 0.f;
      if (on && r < nrows) values8_stats<TYPE>(base + r * rstride, c0, am[u], ss[u]);
    }
    amx = fmaxf(amx, fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])));
    nrm = fmaxf(nrm, warp_sum4(ss, lane));
  }
}
__device__ __forceinline__ void rows_stats_of(int type, const uint8_t* base, long nrows, size_t rstride, int DD,
                                              long gw, long nw, int lane, float& amx, float& nrm) {
  if (type == kTypeQ8) rows_stats<kTypeQ8>(base, nrows, rstride, DD, gw, nw, lane, amx, nrm);
  else if (type == kTypeQ4) rows_stats<kTypeQ4>(base, nrows, rstride, DD, gw, nw, lane, amx, nrm);
  else if (type == kTypeF16) rows_stats<kTypeF16>(base, nrows, rstride, DD, gw, nw, lane, amx, nrm);
  else rows_stats<kTypeF32>(base, nrows, rstride, DD, gw, nw, lane, amx, nrm);
}

// Max |x| and max squared row norm of Q, dO, K^ and V^ (one tensor after the other, every warp of
// the grid taking its share of each), reduced per block.
static __global__ void __launch_bounds__(256) k_row_stats(Params p) {
  __shared__ float red[8][4][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long gw = (long)blockIdx.x * 8 + warp, nw = (long)gridDim.x * 8;
  const long nQ = (long)p.N * p.H, nK = (long)p.M * p.Hkv;
  float amax[4] = {0, 0, 0, 0}, nrm[4] = {0, 0, 0, 0};
  rows_stats<kTypeF32>(reinterpret_cast<const uint8_t*>(p.q), nQ, (size_t)p.D * 4, p.D, gw, nw, lane, amax[0],
                       nrm[0]);
  if (p.dO != nullptr)  // the forward has no dO
    rows_stats<kTypeF32>(reinterpret_cast<const uint8_t*>(p.dO), nQ, (size_t)p.Dv * 4, p.Dv, gw, nw, lane, amax[1],
                         nrm[1]);
  rows_stats_of(p.k_type, p.k, nK, p.rbk, p.D, gw, nw, lane, amax[2], nrm[2]);
  rows_stats_of(p.v_type, p.v, nK, p.rbv, p.Dv, gw, nw, lane, amax[3], nrm[3]);
#pragma unroll
  for (int t = 0; t < 4; ++t) amax[t] = warp_max(amax[t]), nrm[t] = warp_max(nrm[t]);
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
// This warp's keys ja + warp, ja + warp + 8, ... < jb of V^ (head hk), added to acc in key order;
// four keys' loads are issued before their additions.
template <int TYPE>
__device__ __forceinline__ void vsum_keys(const Params& p, int hk, long ja, long jb, int warp, int c0, float* acc) {
  long j = ja + warp;
  for (; j + 24 < jb; j += 32) {
    float x[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) decode8_f<true>(p.v + ((j + 8 * u) * p.Hkv + hk) * p.rbv, TYPE, c0, x[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += x[u][e];
  }
  for (; j < jb; j += 8) {
    float x[8];
    decode8_f<true>(p.v + (j * p.Hkv + hk) * p.rbv, TYPE, c0, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += x[e];
  }
}

static __global__ void __launch_bounds__(256) k_vsum(Params p) {
  // block = (chunk, hk); its eight warps take every eighth key of the chunk and their sums are
  // added in warp order, so the result does not depend on timing
  __shared__ float part[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x / p.Hkv, hk = blockIdx.x % p.Hkv;
  const int c0 = lane * 8;
  const long per = ((long)p.M + p.nbv - 1) / p.nbv;
  const long ja = (long)chunk * per, jb = min((long)p.M, ja + per);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (c0 < p.Dv) {
    if (p.v_type == kTypeQ8) vsum_keys<kTypeQ8>(p, hk, ja, jb, warp, c0, acc);
    else if (p.v_type == kTypeQ4) vsum_keys<kTypeQ4>(p, hk, ja, jb, warp, c0, acc);
    else if (p.v_type == kTypeF16) vsum_keys<kTypeF16>(p, hk, ja, jb, warp, c0, acc);
    else vsum_keys<kTypeF32>(p, hk, ja, jb, warp, c0, acc);
#pragma unroll
    for (int e = 0; e < 8; ++e) part[warp][c0 + e] = acc[e];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < p.Dv; c += 256) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += part[w][c];
    p.vsum[((size_t)chunk * p.Hkv + hk) * p.Dv + c] = t;
  }
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

static __global__ void __launch_bounds__(1024) k_finalize(Params p) {
  __shared__ float am[4], nm[4];
  __shared__ float rn2[1024], ram[1024];
  const int tid = threadIdx.x;
  if (tid < 256) {  // max over the per-block statistics: 32 threads per value, then a warp reduction
    const int q = tid >> 5, lane = tid & 31;  // q = t * 2 + w
    float m = 0.f;
    for (int b = lane; b < p.nblk_stats; b += 32) m = fmaxf(m, p.bstat[(size_t)b * 8 + q]);
    m = warp_max(m);
    if (lane == 0) {
      if ((q & 1) == 0) am[q >> 1] = m;
      else nm[q >> 1] = m;
    }
  }
  // column means of V^ (chunks in order) and max |r|
  float my_am = 0.f;
  const float invM = p.M > 0 ? 1.f / (float)p.M : 0.f;
  for (int idx = tid; idx < p.Hkv * p.Dv; idx += blockDim.x) {
    float s = 0.f;
#pragma unroll 32
    for (int b = 0; b < p.nbv; ++b) s += p.vsum[((size_t)b * p.Hkv) * p.Dv + idx];
    const float r = s * invM;
    p.rmean[idx] = r;
    my_am = fmaxf(my_am, fabsf(r));
  }
  ram[tid] = my_am;
  __syncthreads();
  __shared__ float s_sV, s_utop;
  if (tid == 0) {
    float ramax = 0.f;
    for (int t = 0; t < (int)blockDim.x; ++t) ramax = fmaxf(ramax, ram[t]);
    ram[0] = ramax;
    s_sV = pow2_scale_for(am[3] + ramax, 14);  // |v^ - r| <= |v^| + |r|
    // spacing of binary16 values in the top binade that the shifted operand V' can reach
    int eb = 0;
    frexpf((am[3] + ramax) * s_sV, &eb);  // bound < 2^eb
    s_utop = ldexpf(1.f, eb - 11);
  }
  __syncthreads();
  // The shift actually applied, r', is r rounded (in scaled units) to a multiple of the top
  // binade's spacing, or of binary16's spacing at r where that is coarser.  -r' sV is then an
  // exact binary16 value, and for every cache value whose scaled v^ sV is itself a binary16 value
  // v^ sV - r' sV lands on the binary16 grid: those rows are shifted without rounding.  With r'
  // carrying finer bits, all such values would round by the same amount, an error that does not
  // average out over the keys of a row and that delta (a weighted mean over the keys) keeps whole.
  for (int idx = tid; idx < p.Hkv * p.Dv; idx += blockDim.x) {
    const float x = p.rmean[idx] * s_sV;
    float rs = 0.f;
    if (x != 0.f) {
      int ex = 0;
      frexpf(x, &ex);  // |x| < 2^ex
      const float u = fmaxf(s_utop, ldexpf(1.f, ex - 11));
      rs = rintf(x / u) * u;
    }
    p.rmean[idx] = rs / s_sV;
    p.rsh[idx] = -rs;
  }
  __syncthreads();
  // squared norm of each head's r', taken in a fixed order by one thread per head
  if (tid < p.Hkv && tid < 1024) {
    float n2 = 0.f;
    for (int c = 0; c < p.Dv; ++c) n2 = fmaf(p.rmean[tid * p.Dv + c], p.rmean[tid * p.Dv + c], n2);
    rn2[tid] = n2;
  }
  __syncthreads();
  if (tid == 0) {
    float rmax2 = 0.f;
    const float ramax = ram[0];
    for (int h = 0; h < p.Hkv && h < 1024; ++h) rmax2 = fmaxf(rmax2, rn2[h]);
    Stats s;
    for (int t = 0; t < 4; ++t) s.amax[t] = am[t], s.norm2[t] = nm[t];
    s.rnorm = sqrtf(rmax2);
    s.ramax = ramax;
    s.sQ = pow2_scale_for(am[0], 14);
    s.sdO = pow2_scale_for(am[1], 14);
    s.sK = pow2_scale_for(am[2], 14);
    s.sV = s_sV;
    s.sP = 32768.f;
    // |dP'_ij - delta'_i| <= 2 max_j |dO_i . (v^_j - r)| <= 2 |dO_i| (|v^_j| + |r|), in scaled units
    const float bound = 2.f * (sqrtf(nm[1]) * s.sdO) * ((sqrtf(nm[3]) + s.rnorm) * s.sV) * 1.01f;
    s.lam = pow2_scale_for(bound, 15);
    s.c2 = p.scale * kLog2e / (s.sQ * s.sK);
    s.dq_fac = p.scale / (s.lam * s.sdO * s.sV * s.sK);
    s.dk_fac = p.scale / (s.lam * s.sdO * s.sV * s.sQ);
    s.dv_fac = 1.f / (s.sP * s.sdO);
    s.delta_fac = 1.f / (s.sdO * s.sV);
    s.lamr_exp = ilogbf(s.lam);
    s.cu = p.softcap > 0.f ? p.scale / (p.softcap * s.sQ * s.sK) : 0.f;
    s.cap2 = p.softcap > 0.f ? p.softcap * kLog2e : 0.f;
    *p.st = s;
  }
}

// One warp per (i, h): binary16 rows of Q and dO (row r = i*G + g of head hk), dO_i . r and the
// row's dS multiplier for the dQ product.
static __global__ void __launch_bounds__(256) k_convert(Params p) {
  __shared__ int s_lexp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_lexp = INT_MIN;
  __syncthreads();
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
    if (p.dO == nullptr) continue;  // the forward has no dO
    const float* os = p.dO + rw * p.Dv;
    __half* od = p.do16 + ((size_t)hk * p.R + r) * p.Dv;
    const float* rm = p.rmean + (size_t)hk * p.Dv;
    float dot = 0.f, n2 = 0.f;
    for (int c = 2 * lane; c < p.Dv; c += 64) {
      const float2 x = __ldg(reinterpret_cast<const float2*>(os + c));
      *reinterpret_cast<__half2*>(od + c) = __floats2half2_rn(x.x * sdO, x.y * sdO);
      dot = fmaf(x.x, rm[c], dot);
      dot = fmaf(x.y, rm[c + 1], dot);
      n2 = fmaf(x.x, x.x, fmaf(x.y, x.y, n2));
    }
    dot = warp_sum(dot);
    n2 = warp_sum(n2);
    if (lane == 0) {
      p.dOr[(size_t)hk * p.R + r] = dot;
      // this row's |dS_ij| <= p_ij |dP'_ij - delta'_i| <= 2 |dO_i| max_j |v^_j - r| (scaled units)
      const Stats* st = p.st;
      const float bound = 2.f * (sqrtf(n2) * sdO) * ((sqrtf(st->norm2[3]) + st->rnorm) * st->sV) * 1.01f;
      const float lr = pow2_scale_for(bound, 15);
      p.lamr[(size_t)hk * p.R + r] = lr;
      atomicMax(&s_lexp, ilogbf(lr));
    }
  }
  __syncthreads();
  // the exponents' maximum over rows: the same result in any order
  if (threadIdx.x == 0 && s_lexp != INT_MIN) atomicMax(&p.st->lamr_exp, s_lexp);
}

// One KV head's K' or V' rows (keys 0..M-1 of head hk, DD values each) into the panel-major copy.
// A thread keeps one group of 8 columns, so its V shifts stay in registers, and walks the keys;
// the values are decode8_h's, the rounding of every other decoder.
template <int TYPE>
__device__ __forceinline__ void predecode_head(const Params& p, const uint8_t* base, size_t rb, int DD, float sig,
                                               const float* shift, __half* dst, int hk) {
  const int lg = __ffs(DD / 8) - 1;  // DD / 8 threads per key (a power of two, at most 32)
  const int c0 = (int)(threadIdx.x & ((1u << lg) - 1)) * 8;
  const int kps = 256 >> lg;         // keys per block step
  __half2 sh[4];
  shift8_h(shift, c0, sh);
  __half* d0 = dst + ((size_t)hk * (DD / 64) + c0 / 64) * (size_t)p.M * 64 + (c0 & 63);
  for (long j = (long)blockIdx.x * kps + (threadIdx.x >> lg); j < p.M; j += (long)gridDim.x * kps)
    *reinterpret_cast<uint4*>(d0 + j * 64) = decode8_h_sh(base + ((size_t)j * p.Hkv + hk) * rb, TYPE, c0, sig, sh);
}

// Binary16 operand copies of the cache for the producer-fed passes: K'[hk][j] = k^_j sK and
// V'[hk][j] = v^_j sV - r' sV, with the rounding of the in-kernel decoders (decode8_h), so every
// plan sees the same operands.  The copies are panel-major, [hk][64-column panel][key][64]: the
// TMA box of one operand panel (BK keys x 64 columns) is then one contiguous block.  Grid row
// y < Hkv takes K' of head y, the others V' of head y - Hkv; the cache type is fixed per
// instantiation of the walk.
static __global__ void __launch_bounds__(256) k_predecode(Params p) {
  const bool isv = (int)blockIdx.y >= p.Hkv;
  const int hk = isv ? (int)blockIdx.y - p.Hkv : (int)blockIdx.y;
  const int type = isv ? p.v_type : p.k_type, DD = isv ? p.Dv : p.D;
  const uint8_t* base = isv ? p.v : p.k;
  const size_t rb = isv ? p.rbv : p.rbk;
  const float sig = isv ? p.st->sV : p.st->sK;
  const float* shift = isv ? p.rsh + (size_t)hk * DD : nullptr;
  __half* dst = isv ? p.vd : p.kd;
  if (type == kTypeQ8) predecode_head<kTypeQ8>(p, base, rb, DD, sig, shift, dst, hk);
  else if (type == kTypeQ4) predecode_head<kTypeQ4>(p, base, rb, DD, sig, shift, dst, hk);
  else if (type == kTypeF16) predecode_head<kTypeF16>(p, base, rb, DD, sig, shift, dst, hk);
  else predecode_head<kTypeF32>(p, base, rb, DD, sig, shift, dst, hk);
}

// ------------------------------------------------------------------------------------------------
// row-tile passes: LSE/D statistics (MODE 0) and dQ (MODE 1)
//
// A CTA owns 128 query rows (r = i*G + g of one KV head) and a range of key tiles of BK keys.
// Warp roles (16 warps):
//   warp 0      producer: async copies of raw K/V rows into a ring of `raw_depth` entries
//               (and, in the dQ pass, the TMA load of the Q tile)
//   warp 1      tensor-memory owner and MMA issuer (one lane)
//   warps 4-11  softmax: thread = (row, half of the tile's columns)
//   warps 12-15 decoders: raw rows -> binary16 K' and V' tiles (128-byte swizzled panels)
//   warps 2-3   idle
// Tensor memory: the LSE pass keeps Q and dO there as the A operands of S = Q K'^T and
// dP = dO V'^T; the dQ pass keeps dO there and Q in shared memory, plus the dQ accumulator.
// S and dP have one tensor-memory slot; the softmax warps copy them to registers and release
// the slot at once, so the next tile's products overlap the softmax of this one.

template <int D, int Dv, int BK, int MODE>
struct Rows2Cfg {
  // binary16 K'/V' tile stages: two each where they fit beside the raw ring, else one (the LSE
  // pass at 128 keys x D = 256); the dQ pass keeps one V' stage (its Q tile lives here too)
  static constexpr int KSTAGES = (MODE == 0 && BK * (D + Dv) * 2 * 2 > 160 * 1024) ? 1 : 2;
  static constexpr int VSTAGES = (MODE == 1 || BK * (D + Dv) * 2 * 2 > 160 * 1024) ? 1 : 2;
  static constexpr int QB = MODE ? 128 * D * 2 : 0;
  static constexpr int KB = BK * D * 2, VB = BK * Dv * 2;
  static constexpr int SB = MODE ? 128 * BK * 2 : 0;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + KSTAGES * KB;
  static constexpr int OFF_S = OFF_V + VSTAGES * VB;
  static constexpr int OFF_BAR = OFF_S + SB;
  static constexpr int BAR_BYTES = 2048;  // barriers, tensor-memory slot, LSE merge area
  static constexpr int OFF_RAW = OFF_BAR + BAR_BYTES;
  static constexpr int SMEM_MAX = 232448;
  static constexpr int RAW_BUDGET = SMEM_MAX - 1024 - 64 - OFF_RAW;  // bytes for the raw ring
  // tensor-memory columns; slot s holds S at T_S + 2*BK*s and dP BK columns later
  static constexpr int T_Q = 0;
  static constexpr int T_O = MODE ? 0 : D / 2;
  static constexpr int T_S = T_O + Dv / 2;
  static constexpr int NSLOT = (MODE == 0 && T_S + 4 * BK <= 512) ? 2 : 1;
  static constexpr int T_ACC = T_S + 2 * BK;
  static constexpr int TCOLS = pow2_at_least(MODE ? T_ACC + D : T_S + 2 * BK * NSLOT);
  // softmax warps 4 .. 4+NSOFT-1 (NCH of them per tensor-memory lane quarter, splitting the
  // columns); decoder warps 2, 3 and 4+NSOFT .. 15.  Decoding is the longer of the two per key
  // tile, so one softmax thread per row suffices and ten warps decode.
  static constexpr int NSOFT = 4;
  static constexpr int NCH = NSOFT / 4;
  static constexpr int HALF = BK / NCH;  // columns per softmax thread
  static constexpr int NDEC = 10;
  static constexpr int NT = 32 * (2 + NSOFT + NDEC);  // threads per CTA
};

// barrier indices
constexpr int kMaxRawDepth = 8;  // raw staging entries per tensor
enum {
  B_KRAW_FULL = 0,                            // [kMaxRawDepth] raw K entry landed
  B_KRAW_EMPTY = B_KRAW_FULL + kMaxRawDepth,  // [kMaxRawDepth] raw K entry decoded
  B_VRAW_FULL = B_KRAW_EMPTY + kMaxRawDepth,  // [kMaxRawDepth]
  B_VRAW_EMPTY = B_VRAW_FULL + kMaxRawDepth,  // [kMaxRawDepth]
  B_K_FULL = B_VRAW_EMPTY + kMaxRawDepth,     // [2] K' tile decoded
  B_V_FULL = B_K_FULL + 2,                    // [2] V' tile decoded
  B_K_EMPTY = B_V_FULL + 2,                   // [2] K' tile's products done
  B_V_EMPTY = B_K_EMPTY + 2,                  // [2] V' tile's product done
  B_S_FULL = B_V_EMPTY + 2,                   // [2]
  B_S_FREE = B_S_FULL + 2,                    // [2]
  B_DS_FULL = B_S_FREE + 2,
  B_DS_EMPTY,
  B_ACC_FULL,
  B_Q_FULL,
  B_OPS_READY,
  B_DRAIN0,  // the producer's dQ products, committed after an abort
  B_DRAIN1,  // the issuer's S/dP products, committed after an abort
  B_COUNT
};
static_assert(8 * B_COUNT + 8 <= 512, "barrier area");

struct Waiter {
  volatile int* abort;
  int* err;
  uint64_t limit_ns;
  __device__ __forceinline__ bool operator()(uint64_t* bar, uint32_t parity) const {
    if (mbar_try_wait(bar, parity)) return true;  // fast path: the phase is already complete
    if (*abort) return false;
    if (mbar_wait_bounded(bar, parity, limit_ns)) return true;
    *abort = 1;
    record_error(err, kErrTimeout);
    return false;
  }
};

// ---- leaving after an abort.  A CTA that gave up on a wait still has to let its own
// asynchronous work finish before it frees tensor memory and exits: loads still landing in its
// shared memory, products still reading it.  These waits stop at a deadline too.

// Waits for the phase of `bar` with the given parity until the global timer passes `deadline`.
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && globaltimer_ns() > deadline) return false;
  }
}

// The last loads of a ring of `nst` stages whose full barriers start at `full`, after `issued`
// loads (load n fills stage n % nst and completes phase n / nst of its barrier).  An earlier load
// of a stage has landed: the stage was consumed, and released, before it was refilled.
__device__ __forceinline__ void drain_loads(uint64_t* full, int nst, int issued, uint64_t deadline) {
  for (int n = issued > nst ? issued - nst : 0; n < issued; ++n)
    mbar_wait_until(&full[n % nst], (uint32_t)(n / nst) & 1u, deadline);
}

template <int D, int Dv, int BK, int MODE, bool EXT = false>
static __global__ void __launch_bounds__(Rows2Cfg<D, Dv, BK, MODE>::NT, 1)
    k_rows2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, Params p) {
  using C = Rows2Cfg<D, Dv, BK, MODE>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sS = sm + C::OFF_S;
  uint8_t* sRaw = sm + C::OFF_RAW;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * B_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * B_COUNT + 4);
  float* s_merge = reinterpret_cast<float*>(sm + C::OFF_BAR + 512);  // [128][3]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int r0 = qt * 128;
  const int R = p.R, G = p.G;

  int kt_begin = split * p.kt_per_split;
  int kt_end = min(p.nKT, kt_begin + p.kt_per_split);
  if (p.causal) {
    const long i_hi = (long)min(R - 1, r0 + 127) / G;
    const long jmax = (long)p.M - p.N + i_hi;
    kt_end = min(kt_end, jmax < 0 ? 0 : (int)(jmax / BK) + 1);
  }
  const int ntiles = max(0, kt_end - kt_begin);
  const int KE = p.ke, EPT = BK / KE, RK = p.raw_depth, RV = p.raw_depth_v;
  const int kent = KE * p.rbk_pad, vent = KE * p.rbv_pad;  // bytes of one K / V ring entry
  uint8_t* sRawV = sRaw + RK * kent;

  if (warp == 1) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < kMaxRawDepth; ++s) {
      mbar_init(&bar[B_KRAW_FULL + s], p.raw_bulk ? 1 : 32);
      mbar_init(&bar[B_KRAW_EMPTY + s], C::NDEC);
      mbar_init(&bar[B_VRAW_FULL + s], p.raw_bulk ? 1 : 32);
      mbar_init(&bar[B_VRAW_EMPTY + s], C::NDEC);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_K_FULL + s], C::NDEC);
      mbar_init(&bar[B_V_FULL + s], C::NDEC);
      mbar_init(&bar[B_K_EMPTY + s], 1);
      mbar_init(&bar[B_V_EMPTY + s], 1);
      mbar_init(&bar[B_S_FULL + s], 1);
      mbar_init(&bar[B_S_FREE + s], C::NSOFT);
    }
    mbar_init(&bar[B_DS_FULL], C::NSOFT);
    mbar_init(&bar[B_DS_EMPTY], 1);
    mbar_init(&bar[B_ACC_FULL], 1);
    mbar_init(&bar[B_Q_FULL], 1);
    mbar_init(&bar[B_OPS_READY], C::NSOFT);
    mbar_init(&bar[B_DRAIN0], 1);
    mbar_init(&bar[B_DRAIN1], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  const Stats st = *p.st;
  int n_kraw = 0, n_vraw = 0, n_dq = 0;  // producer: raw entries loaded, dQ products issued
  bool s_issued = false;                 // issuer: any S product issued
  // dQ += dS(t) K'(t) (dQ pass; issued by the producer thread, beside the S/dP stream of warp 1)
  auto issue_dq = [&](int t) {
    if constexpr (MODE != 1) return;  // only the dQ pass has the accumulator and the dS panel
    constexpr uint32_t ID_DQ = idesc_f16(128, D, false, true);
    tc_fence_after();
    const uint64_t da = sdesc_sw128(smem_u32(sS), 16, 1024);
    const uint64_t db = sdesc_sw128(smem_u32(sK + (t % C::KSTAGES) * C::KB), BK * 128, 1024);
#pragma unroll
    for (int k = 0; k < BK / 16; ++k)
      mma_f16(tbase + C::T_ACC, sdesc_adv(da, (k / 4) * (128 * 128) + (k % 4) * 32), sdesc_adv(db, k * 2048), ID_DQ,
              (t > 0 || k > 0) ? 1u : 0u);
    if (t == ntiles - 1) {
      mma_commit(&bar[B_ACC_FULL]);
    } else {
      mma_commit(&bar[B_DS_EMPTY]);
      mma_commit(&bar[B_K_EMPTY + t % C::KSTAGES]);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    // Two rings, one per tensor: entry e of a ring holds keys e*KE .. e*KE+KE-1 of the split.
    // The K and V queues advance independently (whichever has a free slot), so the K rows of
    // the next tile stream in while the V ring waits for the current tile's V' decode.
    if (lane == 0 && p.raw_bulk) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    if (MODE == 1 && lane == 0 && ntiles > 0) {
      mbar_arrive_expect_tx(&bar[B_Q_FULL], (uint32_t)C::QB);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * 128 * 128, &tmQ, &bar[B_Q_FULL], c * 64, r0, hk);
    }
    const int tot = ntiles * EPT;
    int ek = 0, ev = 0, sk = 0, uk = 0, sv = 0, uv = 0;
    uint64_t t0 = globaltimer_ns();
    // one entry of one tensor into its ring slot (bulk: one TMA box of KE rows of this KV head)
    auto load_entry = [&](bool isv, int e, int slot) {
      const int ja = kt_begin * BK + e * KE;
      const int nv = max(0, min(KE, p.M - ja));
      uint64_t* fb = &bar[(isv ? B_VRAW_FULL : B_KRAW_FULL) + slot];
      uint8_t* dst = isv ? sRawV + slot * vent : sRaw + slot * kent;
      const int rb = isv ? p.rbv : p.rbk, rbp = isv ? p.rbv_pad : p.rbk_pad;
      if (p.raw_bulk) {
        if (lane == 0) {
          if (nv > 0) {
            mbar_arrive_expect_tx(fb, (uint32_t)(KE * rb));
            tma_load_3d(dst, isv ? &tmV : &tmK, fb, 0, hk, ja);
          } else {
            mbar_arrive(fb);
          }
        }
      } else {
        const int w = rb / 4;
        const uint8_t* src = isv ? p.v : p.k;
        for (int x = lane; x < nv * w; x += 32) {
          const int rr = x / w, c = x % w;
          cp_async4(dst + rr * rbp + 4 * c, src + ((size_t)(ja + rr) * p.Hkv + hk) * rb + 4 * c);
        }
        cp_async_arrive(fb);
      }
    };
    int nd = 0;  // next dQ product (dQ pass)
    const int ndq = MODE == 1 ? ntiles : 0;
    while (ek < tot || ev < tot || nd < ndq) {
      bool moved = false;
      // the warp takes each decision together (lane 0 polls, the others follow)
      int go_k = 0, go_v = 0, go_q = 0;
      if (lane == 0) {
        go_q = nd < ndq && mbar_try_wait(&bar[B_DS_FULL], nd & 1);
        go_k = ek < tot && mbar_try_wait(&bar[B_KRAW_EMPTY + sk], (uk & 1) ^ 1);
        go_v = ev < tot && mbar_try_wait(&bar[B_VRAW_EMPTY + sv], (uv & 1) ^ 1);
      }
      go_q = __shfl_sync(0xffffffffu, go_q, 0);
      go_k = __shfl_sync(0xffffffffu, go_k, 0);
      go_v = __shfl_sync(0xffffffffu, go_v, 0);
      if (go_q) {
        if (lane == 0) issue_dq(nd);
        __syncwarp();
        ++nd;
        moved = true;
      }
      if (go_v) {
        load_entry(true, ev, sv);
        ++ev;
        if (++sv == RV) sv = 0, ++uv;
        moved = true;
      }
      if (go_k) {
        load_entry(false, ek, sk);
        ++ek;
        if (++sk == RK) sk = 0, ++uk;
        moved = true;
      }
      if (moved) {
        t0 = globaltimer_ns();
      } else {
        if (*s_abort) break;
        if (globaltimer_ns() - t0 > p.wait_ns) {
          if (lane == 0) {
            *s_abort = 1;
            record_error(p.err, kErrTimeout);
          }
          break;
        }
        __nanosleep(64);
      }
    }
    n_kraw = ek, n_vraw = ev, n_dq = nd;
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
      const uint32_t tQ = tbase + C::T_Q, tO = tbase + C::T_O;
      const bool ok = (MODE == 0 || wait(&bar[B_Q_FULL], 0)) && wait(&bar[B_OPS_READY], 0);
      // S(t) = Q K'^T into the tensor-memory slot of tile t
      auto issue_s = [&](int t) {
        const uint32_t tS = tbase + C::T_S + 2 * BK * (t % C::NSLOT);
        s_issued = true;
        tc_fence_after();
        const uint64_t db = sdesc_sw128(smem_u32(sK + (t % C::KSTAGES) * C::KB), 16, 1024);
        const uint64_t da = sdesc_sw128(smem_u32(sQ), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t bd = sdesc_adv(db, (k / 4) * (BK * 128) + (k % 4) * 32);
          if (MODE == 1)
            mma_f16(tS, sdesc_adv(da, (k / 4) * (128 * 128) + (k % 4) * 32), bd, ID_S, k > 0);
          else
            mma_f16_tmem_a(tS, tQ + k * 8, bd, ID_S, k > 0);
        }
        if (MODE == 0) mma_commit(&bar[B_K_EMPTY + t % C::KSTAGES]);  // K' of tile t is not read again
      };
      // dP(t) = dO V'^T next to S(t); the slot is then complete
      auto issue_dp = [&](int t) {
        const int vs = t % C::VSTAGES, sl = t % C::NSLOT;
        const uint32_t tP = tbase + C::T_S + 2 * BK * sl + BK;
        tc_fence_after();
        const uint64_t dv = sdesc_sw128(smem_u32(sV + vs * C::VB), 16, 1024);
#pragma unroll
        for (int k = 0; k < Dv / 16; ++k)
          mma_f16_tmem_a(tP, tO + k * 8, sdesc_adv(dv, (k / 4) * (BK * 128) + (k % 4) * 32), ID_S, k > 0);
        mma_commit(&bar[B_S_FULL + sl]);
        mma_commit(&bar[B_V_EMPTY + vs]);
      };
      if (MODE == 0) {
        for (int t = 0; ok && t < ntiles; ++t) {
          const int su = t / C::NSLOT;
          if (!wait(&bar[B_K_FULL + t % C::KSTAGES], (t / C::KSTAGES) & 1) ||
              !wait(&bar[B_S_FREE + t % C::NSLOT], (su & 1) ^ 1))
            break;
          issue_s(t);
          if (!wait(&bar[B_V_FULL + t % C::VSTAGES], (t / C::VSTAGES) & 1)) break;
          issue_dp(t);
        }
      } else if (ok) {
        // S(t) and dP(t) in order; the dQ products are issued by the producer thread
        for (int t = 0; t < ntiles; ++t) {
          if (!wait(&bar[B_K_FULL + t % C::KSTAGES], (t / C::KSTAGES) & 1) || !wait(&bar[B_S_FREE], (t & 1) ^ 1))
            break;
          issue_s(t);
          if (!wait(&bar[B_V_FULL + t % C::VSTAGES], (t / C::VSTAGES) & 1)) break;
          issue_dp(t);
        }
      }
    }
  } else if (warp >= 4 + C::NSOFT || warp == 2 || warp == 3) {
    // ------------------------------------------------------------------ decoders
    // Per tile: the K' rows of all its entries, then (once the previous dP has released the
    // V' stage) the V' rows.
    constexpr int NDT = C::NDEC * 32;
    static_assert(NDT % 64 == 0, "decoder_map needs a multiple of 8 column groups of 8 lanes");
    const int dt = (warp < 4 ? warp - 2 : warp - (4 + C::NSOFT) + 2) * 32 + lane;
    __half2 vsh[16];
    load_group_shift<Dv, NDT>(p.rsh + (size_t)hk * Dv, p.v_type, dt, vsh);
    int sk = 0, uk = 0, sv = 0, uv = 0;  // ring positions
    bool ok = true;
    for (int t = 0; ok && t < ntiles; ++t) {
      const int ks = t % C::KSTAGES, vs = t % C::VSTAGES;
      const int j0 = (kt_begin + t) * BK;
      if (!wait(&bar[B_K_EMPTY + ks], ((t / C::KSTAGES) & 1) ^ 1)) break;
      const uint32_t kd = smem_u32(sK + ks * C::KB), vd = smem_u32(sV + vs * C::VB);
      for (int h = 0; h < EPT; ++h) {
        if (!(ok = wait(&bar[B_KRAW_FULL + sk], uk & 1))) break;
        const int nv = max(0, min(KE, p.M - (j0 + h * KE)));
        decode_rows<D, BK, NDT, false>(p.k_type, smem_u32(sRaw) + sk * kent, p.rbk_pad, KE, nv, h * KE, kd, st.sK,
                                       vsh, dt);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_KRAW_EMPTY + sk]);  // raw entry consumed
        if (++sk == RK) sk = 0, ++uk;
      }
      if (!ok) break;
      fence_proxy_async_smem();  // the tile's binary16 stores, visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_K_FULL + ks]);
      if (!wait(&bar[B_V_EMPTY + vs], ((t / C::VSTAGES) & 1) ^ 1)) break;
      for (int h = 0; h < EPT; ++h) {
        if (!(ok = wait(&bar[B_VRAW_FULL + sv], uv & 1))) break;
        const int nv = max(0, min(KE, p.M - (j0 + h * KE)));
        decode_rows<Dv, BK, NDT, true>(p.v_type, smem_u32(sRawV) + sv * vent, p.rbv_pad, KE, nv, h * KE, vd,
                                       st.sV, vsh, dt);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_VRAW_EMPTY + sv]);
        if (++sv == RV) sv = 0, ++uv;
      }
      if (!ok) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_V_FULL + vs]);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax
    const int q4 = warp & 3, ch = (warp - 4) >> 2;  // ch < C::NCH
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int r = r0 + row;
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
    // the dQ pass scales this row's dS by its own power of two lamr (the product sums over keys only)
    const float lam = (MODE == 1 && rvalid) ? p.lamr[(size_t)hk * R + r] : st.lam;
    const float c2 = st.c2, dq_fac = st.dq_fac * (st.lam / lam);
    // 2^(t2 + nlse2) = p (0 on a dead row); in the dQ pass the exponent also carries log2(lam),
    // so the exponential yields lam * p directly (lam is a power of two)
    const float nlse2 = live ? -lse2 + (MODE == 1 ? (float)ilogbf(lam) : 0.f) : -CUDART_INF_F;
    const uint32_t sS_u = smem_u32(sS);
    float m2 = -CUDART_INF_F, l = 0.f, lc = 0.f, sd = 0.f, sdc = 0.f;

    if (ntiles > 0) {
      // this thread's share of the row's A operands into tensor memory (binary16 pairs per column)
      auto put_row = [&](const __half* src, int DD, uint32_t tcol) {
        // DD/2 32-bit words per row, split between the NCH threads of the row; a share under
        // 32 words goes whole to the first (tensor-memory stores move 32 columns at a time)
        const int wpr = DD / 2;
        const int per = wpr / C::NCH;
        const int w0 = per >= 32 ? ch * per : 0, nw = per >= 32 ? per : (ch == 0 ? wpr : 0);
        const uint4* s4 = reinterpret_cast<const uint4*>(src) + w0 / 4;
        for (int c = 0; c < nw; c += 32) {
          uint32_t wv[32];
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const uint4 u = rvalid ? __ldg(s4 + c / 4 + x) : make_uint4(0, 0, 0, 0);
            wv[4 * x] = u.x, wv[4 * x + 1] = u.y, wv[4 * x + 2] = u.z, wv[4 * x + 3] = u.w;
          }
          tmem_st32(tbase + lane_off + tcol + w0 + c, wv);
        }
      };
      const size_t rowq = (size_t)hk * R + (rvalid ? r : 0);
      if (MODE == 0) put_row(p.q16 + rowq * D, D, C::T_Q);
      put_row(p.do16 + rowq * Dv, Dv, C::T_O);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_OPS_READY]);
    }

    for (int t = 0; t < ntiles; ++t) {
      const int j0 = (kt_begin + t) * BK;
      const int sl = t % C::NSLOT, su = t / C::NSLOT;
      if (!wait(&bar[B_S_FULL + sl], su & 1)) break;
      tc_fence_after();
      bool stored_wait = false;
      const uint32_t tS = tbase + C::T_S + 2 * BK * sl;
#pragma unroll 1
      for (int c = 0; c < C::HALF; c += 32) {
        const int col0 = ch * C::HALF + c;
        float s[32], dp[32];
        tmem_ld32(tS + lane_off + col0, s);
        tmem_ld32(tS + BK + lane_off + col0, dp);
        tmem_ld_wait();
        if (c + 32 >= C::HALF) {  // the slot is free once its last columns are in registers
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[B_S_FREE + sl]);
        }
        // fully visible chunk without a mask: no per-key tests
        const bool full = mrow == nullptr && (long)(j0 + col0 + 31) <= jlast;
        float t2[32];  // log2-domain scores (dQ pass: already minus lse, plus log2(lam))
        const float t2off = MODE == 1 ? nlse2 : 0.f;
        if constexpr (EXT) {
#pragma unroll
          for (int n = 0; n < 32; ++n) t2[n] = s[n];
          ext_scores<MODE == 1 ? 1 : 0>(t2, nullptr, j0 + col0, r, hk, t2off, 0.f, jlast, mrow, st, p.alibi, G,
                                        p.M - p.N);
        } else if (full) {
#pragma unroll
          for (int n = 0; n < 32; ++n) t2[n] = fmaf(s[n], c2, t2off);
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            const int j = j0 + col0 + n;
            bool ok = (long)j <= jlast;
            float mv = 0.f;
            if (ok && mrow) {
              mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
              ok = !(mv == -CUDART_INF_F);
            }
            t2[n] = ok ? fmaf(s[n], c2, fmaf(mv, kLog2e, t2off)) : -CUDART_INF_F;
          }
        }
        if (MODE == 0) {
          float cmax = -CUDART_INF_F;
#pragma unroll
          for (int n = 0; n < 32; ++n) cmax = fmaxf(cmax, t2[n]);
          if (cmax > m2) {
            const float f = ex2(m2 - cmax);  // 0 while m2 = -inf
            l *= f, lc *= f, sd *= f, sdc *= f;
            m2 = cmax;
          }
          if (cmax > -CUDART_INF_F) {
            float cl = 0.f, cs = 0.f;
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              const float e = ex2(t2[n] - m2);
              cl += e;
              cs = fmaf(e, dp[n], cs);
            }
            // compensated accumulation of the chunk sums
            float y = cl - lc, tt = l + y;
            lc = (tt - l) - y, l = tt;
            y = cs - sdc, tt = sd + y;
            sdc = (tt - sd) - y, sd = tt;
          }
        } else {
          uint32_t pk[16];
#pragma unroll
          for (int n = 0; n < 32; n += 2) {
            const float p0 = ex2(t2[n]), p1 = ex2(t2[n + 1]);  // lam * p; 0 for masked keys, dead rows
            pk[n / 2] = h2_as_u32(__floats2half2_rn(p0 * (dp[n] - dl), p1 * (dp[n + 1] - dl)));
          }
          if (!stored_wait) {
            if (!wait(&bar[B_DS_EMPTY], (t & 1) ^ 1)) break;
            stored_wait = true;
          }
#pragma unroll
          for (int x = 0; x < 4; ++x)
            sts_v4(sS_u + panel_off_u(128, row, col0 + 8 * x), pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
      }
      if (*s_abort) break;
      if (MODE == 1) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_DS_FULL]);
      }
    }

    // epilogue
    if (MODE == 0) {
      if (C::NCH == 2) {
        if (ch == 1) s_merge[row * 3 + 0] = m2, s_merge[row * 3 + 1] = l, s_merge[row * 3 + 2] = sd;
        named_bar_sync(1, 32 * C::NSOFT);
      }
      if (ch == 0 && rvalid) {
        float m2b = -CUDART_INF_F, lb = 0.f, sdb = 0.f;
        if (C::NCH == 2) m2b = s_merge[row * 3 + 0], lb = s_merge[row * 3 + 1], sdb = s_merge[row * 3 + 2];
        const float mm = fmaxf(m2, m2b);
        float L = 0.f, SD = 0.f;
        if (mm > -CUDART_INF_F) {
          const float fa = ex2(m2 - mm), fb = ex2(m2b - mm);
          L = l * fa + lb * fb;
          SD = sd * fa + sdb * fb;
        }
        float* o = p.part + (((size_t)split * p.Hkv + hk) * R + r) * 3;
        o[0] = mm, o[1] = L, o[2] = SD;
      }
    } else {
      float* out = !rvalid ? nullptr
                   : p.nsplit == 1 ? p.dQ + ((size_t)i * p.H + h) * D
                                   : p.dqpart + (((size_t)split * p.Hkv + hk) * R + r) * D;
      const bool have = ntiles > 0 && wait(&bar[B_ACC_FULL], 0);
      if (have) tc_fence_after();
#pragma unroll 1
      for (int c = ch * (D / C::NCH); c < (ch + 1) * (D / C::NCH); c += 32) {
        float v[32];
        if (have) {
          tmem_ld32(tbase + C::T_ACC + lane_off + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (out) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(out + c + e) =
                make_float4(v[e] * dq_fac, v[e + 1] * dq_fac, v[e + 2] * dq_fac, v[e + 3] * dq_fac);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (warp == 0 && lane == 0) {
      drain_loads(&bar[B_KRAW_FULL], RK, n_kraw, deadline);
      drain_loads(&bar[B_VRAW_FULL], RV, n_vraw, deadline);
      if (MODE == 1 && ntiles > 0) mbar_wait_until(&bar[B_Q_FULL], 0, deadline);
      if (n_dq > 0) {
        mma_commit(&bar[B_DRAIN0]);
        mbar_wait_until(&bar[B_DRAIN0], 0, deadline);
      }
    }
    if (warp == 1 && lane == 0 && s_issued) {
      mma_commit(&bar[B_DRAIN1]);
      mbar_wait_until(&bar[B_DRAIN1], 0, deadline);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// ------------------------------------------------------------------------------------------------
// producer-fed row passes: the LSE/D pass (MODE 0) and the dQ pass (MODE 1) over the binary16
// K'/V' copies written by k_predecode, which arrive as 128-byte-swizzled TMA panels.  With no
// decoding inside the CTA, the operand stages take the shared memory the raw rings held.
//
// Warp roles: warp 0 producer (TMA loads of K'/V' tiles and, in the dQ pass, of the Q tile; it
// also issues the dQ products), warp 1 tensor-memory owner and S/dP issuer, warps 2.. softmax:
// four per 32-key chunk of the tile (one per tensor-memory lane quarter), so a softmax thread
// owns one row and one chunk.  S and dP each have a full/free barrier pair; the softmax frees
// S as soon as its chunk is in registers, so S(t+1) is computed while dP(t) is still read.

template <int D, int Dv, int BK, int MODE>
struct Rows3Cfg {
  // MODE 0: LSE/D pass; 1: dQ pass
  static_assert(MODE == 0 || MODE == 1, "pass");
  static constexpr bool ROWQ = MODE == 1;  // Q tile in shared memory; a product over the row's dS panel
  static constexpr int QB = ROWQ ? 128 * D * 2 : 0;
  static constexpr int KB = BK * D * 2, VB = BK * Dv * 2;
  static constexpr int SB = ROWQ ? 128 * BK * 2 : 0;
  static constexpr int NCH = BK / 32;  // 32-key chunks per tile
  static constexpr int NSOFT = 4 * NCH;
  // dP is issued by a thread of its own (after the softmax warps), so one issuing thread's waits
  // and commits run while the other's products keep the pipe fed.  In the LSE pass the two take
  // turns, S(t), dP(t), S(t+1), ..., each waiting for the other's products of the previous step to
  // be issued: left free, S ran ahead of dP, which waits for the single V' stage
  static constexpr bool DP_OWN = true;
  static constexpr bool ALT = MODE == 0;
  static constexpr int W_DP = 2 + NSOFT;
  static constexpr int NT = 32 * (2 + NSOFT + (DP_OWN ? 1 : 0));
  static constexpr int MERGE_BYTES = MODE == 0 ? (NCH - 1) * 128 * 3 * 4 : 0;
  static constexpr int BAR_BYTES = 512 + MERGE_BYTES;
  static constexpr int SMEM_MAX = 232448;
  static constexpr int AVAIL = SMEM_MAX - 1024 - BAR_BYTES - QB - SB;
  // K'/V' stages (at most 4 each): K first, then alternately, while they fit
  static constexpr int stage_pair() {
    int k = 1, v = 1;
    for (;;) {
      if (k <= v && k < 4 && (k + 1) * KB + v * VB <= AVAIL)
        ++k;
      else if (v < k && v < 4 && k * KB + (v + 1) * VB <= AVAIL)
        ++v;
      else if (k < 4 && (k + 1) * KB + v * VB <= AVAIL)
        ++k;
      else
        break;
    }
    return k * 8 + v;
  }
  static constexpr int KSTAGES = stage_pair() / 8, VSTAGES = stage_pair() % 8;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + KSTAGES * KB;
  static constexpr int OFF_S = OFF_V + VSTAGES * VB;
  static constexpr int OFF_BAR = OFF_S + SB;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + 1024 for aligning the base
  // tensor-memory columns: [Q' (LSE/D pass)] [dO'] [S] [dP] [dQ accumulator (dQ pass)]
  static constexpr int T_Q = 0;
  static constexpr int T_O = ROWQ ? 0 : D / 2;
  static constexpr int T_S = T_O + Dv / 2;
  static constexpr int T_P = T_S + BK;
  static constexpr int T_ACC = T_P + BK;
  static constexpr int ACC_N = ROWQ ? D : 0;  // accumulator columns
  static constexpr int TCOLS = pow2_at_least(T_ACC + ACC_N);
  static_assert(KB + VB <= AVAIL && SMEM <= SMEM_MAX, "shared memory budget");
  static_assert(TCOLS <= 512, "tensor memory budget");
  static_assert(BK % 32 == 0 && BK <= 128, "key tile");
};

enum {
  R3_K_FULL = 0,   // [4] K' tile landed
  R3_K_EMPTY = 4,  // [4] K' tile's products done
  R3_V_FULL = 8,   // [4]
  R3_V_EMPTY = 12,  // [4]
  R3_S_FULL = 16,
  R3_S_FREE,
  R3_P_FULL,
  R3_P_FREE,
  R3_DS_FULL,
  R3_DS_EMPTY,
  R3_ACC_FULL,
  R3_Q_FULL,
  R3_OPS_READY,
  R3_DRAIN0,  // the producer's dQ products, committed after an abort
  R3_DRAIN1,  // the S/dP issuer's products, committed after an abort
  R3_DRAIN2,  // the dP issuer's products, committed after an abort
  R3_S_ISSUED,   // S(t) issued (LSE pass: the dP thread's turn)
  R3_DP_ISSUED,  // dP(t) issued (LSE pass: the S thread's turn)
  R3_COUNT
};
static_assert(8 * R3_COUNT + 8 <= 512, "barrier area");

template <int D, int Dv, int BK, int MODE, bool EXT = false>
static __global__ void __launch_bounds__(Rows3Cfg<D, Dv, BK, MODE>::NT, 1)
    k_rows3(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, Params p) {
  using C = Rows3Cfg<D, Dv, BK, MODE>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sS = sm + C::OFF_S;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * R3_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * R3_COUNT + 4);
  float* s_merge = reinterpret_cast<float*>(sm + C::OFF_BAR + 512);  // [NCH-1][128][3]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int r0 = qt * 128;
  const int R = p.R, G = p.G;

  const int kt_begin = split * p.kt_per_split;
  int kt_end = min(p.nKT, kt_begin + p.kt_per_split);
  if (p.causal) {
    const long i_hi = (long)min(R - 1, r0 + 127) / G;
    const long jmax = (long)p.M - p.N + i_hi;
    kt_end = min(kt_end, jmax < 0 ? 0 : (int)(jmax / BK) + 1);
  }
  const int ntiles = max(0, kt_end - kt_begin);

  if (warp == 1) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar[R3_K_FULL + s], 1);
      mbar_init(&bar[R3_K_EMPTY + s], 1);
      mbar_init(&bar[R3_V_FULL + s], 1);
      mbar_init(&bar[R3_V_EMPTY + s], 1);
    }
    mbar_init(&bar[R3_S_FULL], 1);
    mbar_init(&bar[R3_S_FREE], C::NSOFT);
    mbar_init(&bar[R3_P_FULL], 1);
    mbar_init(&bar[R3_P_FREE], C::NSOFT);
    mbar_init(&bar[R3_DS_FULL], C::NSOFT);
    mbar_init(&bar[R3_DS_EMPTY], 1);
    mbar_init(&bar[R3_ACC_FULL], 1);
    mbar_init(&bar[R3_Q_FULL], 1);
    mbar_init(&bar[R3_OPS_READY], C::NSOFT);
    mbar_init(&bar[R3_DRAIN0], 1);
    mbar_init(&bar[R3_DRAIN1], 1);
    mbar_init(&bar[R3_DRAIN2], 1);
    mbar_init(&bar[R3_S_ISSUED], 1);
    mbar_init(&bar[R3_DP_ISSUED], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  const Stats st = *p.st;
  int n_kload = 0, n_vload = 0, n_prod = 0;  // producer: K' and V' tiles loaded, products issued
  bool s_issued = false;                     // an issuer: any product issued

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      if (C::ROWQ && ntiles > 0) {
        mbar_arrive_expect_tx(&bar[R3_Q_FULL], (uint32_t)C::QB);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * 128 * 128, &tmQ, &bar[R3_Q_FULL], c * 64, r0, hk);
      }
      // the dQ pass's product over the row tile's dS panel, beside the S/dP stream of warp 1:
      // dQ += dS(t) K'(t); it frees the K' stage it read
      auto issue_dq = [&](int t) {
        if constexpr (C::ROWQ) {
          constexpr uint32_t ID_A = idesc_f16(128, D, false, true);
          tc_fence_after();
          const uint64_t da = sdesc_sw128(smem_u32(sS), 16, 1024);
          const uint64_t db = sdesc_sw128(smem_u32(sK + (t % C::KSTAGES) * C::KB), BK * 128, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16(tbase + C::T_ACC, sdesc_adv(da, (k / 4) * (128 * 128) + (k % 4) * 32), sdesc_adv(db, k * 2048),
                    ID_A, (t > 0 || k > 0) ? 1u : 0u);
          if (t == ntiles - 1) {
            mma_commit(&bar[R3_ACC_FULL]);
          } else {
            mma_commit(&bar[R3_DS_EMPTY]);
            mma_commit(&bar[R3_K_EMPTY + t % C::KSTAGES]);
          }
        }
      };
      const int ndq = C::ROWQ ? ntiles : 0, nvt = ntiles;
      int kt = 0, vt = 0, nd = 0;
      uint64_t t0 = globaltimer_ns();
      while (kt < ntiles || vt < nvt || nd < ndq) {
        bool moved = false;
        if (nd < ndq && mbar_try_wait(&bar[R3_DS_FULL], nd & 1)) {
          issue_dq(nd);
          ++nd;
          moved = true;
        }
        if (kt < ntiles && mbar_try_wait(&bar[R3_K_EMPTY + kt % C::KSTAGES], ((kt / C::KSTAGES) & 1) ^ 1)) {
          uint64_t* fb = &bar[R3_K_FULL + kt % C::KSTAGES];
          uint8_t* dst = sK + (kt % C::KSTAGES) * C::KB;
          const int j0 = (kt_begin + kt) * BK;
          mbar_arrive_expect_tx(fb, (uint32_t)C::KB);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * BK * 128, &tmK, fb, 0, j0, hk * (D / 64) + c);
          ++kt;
          moved = true;
        }
        if (vt < nvt && mbar_try_wait(&bar[R3_V_EMPTY + vt % C::VSTAGES], ((vt / C::VSTAGES) & 1) ^ 1)) {
          uint64_t* fb = &bar[R3_V_FULL + vt % C::VSTAGES];
          uint8_t* dst = sV + (vt % C::VSTAGES) * C::VB;
          const int j0 = (kt_begin + vt) * BK;
          mbar_arrive_expect_tx(fb, (uint32_t)C::VB);
#pragma unroll
          for (int c = 0; c < Dv / 64; ++c) tma_load_3d(dst + c * BK * 128, &tmV, fb, 0, j0, hk * (Dv / 64) + c);
          ++vt;
          moved = true;
        }
        if (moved) {
          t0 = globaltimer_ns();
        } else {
          if (*s_abort) break;
          if (globaltimer_ns() - t0 > p.wait_ns) {
            *s_abort = 1;
            record_error(p.err, kErrTimeout);
            break;
          }
        }
      }
      n_kload = kt, n_vload = vt, n_prod = nd;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S/dP issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
      const uint32_t tQ = tbase + C::T_Q, tO = tbase + C::T_O;
      const uint32_t tS = tbase + C::T_S, tP = tbase + C::T_P;
      const bool ok = (!C::ROWQ || wait(&bar[R3_Q_FULL], 0)) && wait(&bar[R3_OPS_READY], 0);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int ks = t % C::KSTAGES, vs = t % C::VSTAGES;
        if (!wait(&bar[R3_K_FULL + ks], (t / C::KSTAGES) & 1) || !wait(&bar[R3_S_FREE], (t & 1) ^ 1)) break;
        if (C::ALT && t > 0 && !wait(&bar[R3_DP_ISSUED], (t - 1) & 1)) break;
        s_issued = true;
        tc_fence_after();
        const uint64_t db = sdesc_sw128(smem_u32(sK + ks * C::KB), 16, 1024);
        const uint64_t da = sdesc_sw128(smem_u32(sQ), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t bd = sdesc_adv(db, (k / 4) * (BK * 128) + (k % 4) * 32);
          if (C::ROWQ)
            mma_f16(tS, sdesc_adv(da, (k / 4) * (128 * 128) + (k % 4) * 32), bd, ID_S, k > 0);
          else
            mma_f16_tmem_a(tS, tQ + k * 8, bd, ID_S, k > 0);
        }
        mma_commit(&bar[R3_S_FULL]);
        if (!C::ROWQ) mma_commit(&bar[R3_K_EMPTY + ks]);  // only the dQ pass reads K'(t) again
        if (C::ALT) mbar_arrive(&bar[R3_S_ISSUED]);
        if constexpr (!C::DP_OWN) {
          if (!wait(&bar[R3_V_FULL + vs], (t / C::VSTAGES) & 1) || !wait(&bar[R3_P_FREE], (t & 1) ^ 1)) break;
          tc_fence_after();
          const uint64_t dv = sdesc_sw128(smem_u32(sV + vs * C::VB), 16, 1024);
#pragma unroll
          for (int k = 0; k < Dv / 16; ++k)
            mma_f16_tmem_a(tP, tO + k * 8, sdesc_adv(dv, (k / 4) * (BK * 128) + (k % 4) * 32), ID_S, k > 0);
          mma_commit(&bar[R3_P_FULL]);
          mma_commit(&bar[R3_V_EMPTY + vs]);
        }
      }
    }
  } else if (C::DP_OWN && warp == C::W_DP) {
    // ------------------------------------------------------------------ dP issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
      const uint32_t tO = tbase + C::T_O, tP = tbase + C::T_P;
      const bool ok = wait(&bar[R3_OPS_READY], 0);  // dO' in tensor memory
      for (int t = 0; ok && t < ntiles; ++t) {
        const int vs = t % C::VSTAGES;
        if (C::ALT && !wait(&bar[R3_S_ISSUED], t & 1)) break;
        if (!wait(&bar[R3_V_FULL + vs], (t / C::VSTAGES) & 1) || !wait(&bar[R3_P_FREE], (t & 1) ^ 1)) break;
        s_issued = true;
        tc_fence_after();
        const uint64_t dv = sdesc_sw128(smem_u32(sV + vs * C::VB), 16, 1024);
#pragma unroll
        for (int k = 0; k < Dv / 16; ++k)
          mma_f16_tmem_a(tP, tO + k * 8, sdesc_adv(dv, (k / 4) * (BK * 128) + (k % 4) * 32), ID_S, k > 0);
        mma_commit(&bar[R3_P_FULL]);
        mma_commit(&bar[R3_V_EMPTY + vs]);
        if (C::ALT) mbar_arrive(&bar[R3_DP_ISSUED]);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax
    const int q4 = warp & 3, ch = (warp - 2) >> 2;  // ch < C::NCH
    const int row = q4 * 32 + lane;
    const int col0 = ch * 32;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int r = r0 + row;
    const bool rvalid = r < R;
    const int i = rvalid ? r / G : 0;
    const int h = hk * G + (rvalid ? r % G : 0);
    const long jlast = rvalid ? (p.causal ? min((long)p.M - 1, (long)p.M - p.N + i) : (long)p.M - 1) : -1;
    const uint16_t* mrow = p.mask ? p.mask + ((size_t)(h % p.Hm) * p.N + i) * p.M : nullptr;
    float lse2 = -CUDART_INF_F, dl = 0.f;
    if (C::ROWQ && rvalid) {
      lse2 = p.lse2[(size_t)hk * R + r];
      dl = p.dlt[(size_t)hk * R + r];
    }
    const bool live = C::ROWQ ? (lse2 > -CUDART_INF_F) : rvalid;
    // the dQ pass scales this row's dS by its own power of two lamr (the product sums over keys only)
    const float lam = (C::ROWQ && rvalid) ? p.lamr[(size_t)hk * R + r] : st.lam;
    const float c2 = st.c2, dq_fac = st.dq_fac * (st.lam / lam);
    // 2^(t2 + nlse2) = p (0 on a dead row); the exponent also carries log2 of the power-of-two
    // multiplier lam of the dS panel, so the exponential yields lam * p directly
    // (dS = lam p (dP - delta))
    const float nlse2 = live ? -lse2 + (float)ilogbf(lam) : -CUDART_INF_F;
    const float t2off = C::ROWQ ? nlse2 : 0.f;
    const uint32_t sS_u = smem_u32(sS);
    float m2 = -CUDART_INF_F, l = 0.f, lc = 0.f, sd = 0.f, sdc = 0.f;

    if (ntiles > 0) {
      // this thread's share of the row's A operands into tensor memory (binary16 pairs per column)
      auto put_row = [&](const __half* src, int DD, uint32_t tcol) {
        const int wpr = DD / 2;
        const int per = wpr / C::NCH;
        const int w0 = per >= 32 ? ch * per : 0, nw = per >= 32 ? per : (ch == 0 ? wpr : 0);
        const uint4* s4 = reinterpret_cast<const uint4*>(src) + w0 / 4;
        for (int c = 0; c < nw; c += 32) {
          uint32_t wv[32];
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const uint4 u = rvalid ? __ldg(s4 + c / 4 + x) : make_uint4(0, 0, 0, 0);
            wv[4 * x] = u.x, wv[4 * x + 1] = u.y, wv[4 * x + 2] = u.z, wv[4 * x + 3] = u.w;
          }
          tmem_st32(tbase + lane_off + tcol + w0 + c, wv);
        }
      };
      const size_t rowq = (size_t)hk * R + (rvalid ? r : 0);
      if (!C::ROWQ) put_row(p.q16 + rowq * D, D, C::T_Q);
      put_row(p.do16 + rowq * Dv, Dv, C::T_O);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[R3_OPS_READY]);
    }

    for (int t = 0; t < ntiles; ++t) {
      const int j0 = (kt_begin + t) * BK;
      float s[32], dp[32];
      if (!wait(&bar[R3_S_FULL], t & 1)) break;
      tc_fence_after();
      tmem_ld32(tbase + C::T_S + lane_off + col0, s);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[R3_S_FREE]);
      // log2-domain scores (dQ pass: already minus lse, plus log2(lam)); masked keys -> -inf
      if constexpr (EXT) {
        ext_scores<MODE>(s, nullptr, j0 + col0, r, hk, t2off, 0.f, jlast, mrow, st, p.alibi, G,
                                      p.M - p.N);
      } else if (mrow == nullptr && (long)(j0 + col0 + 31) <= jlast) {
#pragma unroll
        for (int n = 0; n < 32; ++n) s[n] = fmaf(s[n], c2, t2off);
      } else {
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          const int j = j0 + col0 + n;
          bool ok = (long)j <= jlast;
          float mv = 0.f;
          if (ok && mrow) {
            mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
            ok = !(mv == -CUDART_INF_F);
          }
          s[n] = ok ? fmaf(s[n], c2, fmaf(mv, kLog2e, t2off)) : -CUDART_INF_F;
        }
      }
      bool any = true;
      if (!C::ROWQ) {
        float cmax = -CUDART_INF_F;
#pragma unroll
        for (int n = 0; n < 32; ++n) cmax = fmaxf(cmax, s[n]);
        if (cmax > m2) {
          const float f = ex2(m2 - cmax);  // 0 while m2 = -inf
          l *= f, lc *= f, sd *= f, sdc *= f;
          m2 = cmax;
        }
        any = cmax > -CUDART_INF_F;
        if (any) {
#pragma unroll
          for (int n = 0; n < 32; ++n) s[n] = ex2(s[n] - m2);
        }
      } else {
#pragma unroll
        for (int n = 0; n < 32; ++n) s[n] = ex2(s[n]);  // lam * p; 0 for masked keys, dead rows
      }
      if (!wait(&bar[R3_P_FULL], t & 1)) break;
      tc_fence_after();
      tmem_ld32(tbase + C::T_P + lane_off + col0, dp);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[R3_P_FREE]);
      if (!C::ROWQ) {
        if (any) {
          float cl = 0.f, cs = 0.f;
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            cl += s[n];
            cs = fmaf(s[n], dp[n], cs);
          }
          // compensated accumulation of the chunk sums
          float y = cl - lc, tt = l + y;
          lc = (tt - l) - y, l = tt;
          y = cs - sdc, tt = sd + y;
          sdc = (tt - sd) - y, sd = tt;
        }
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int n = 0; n < 32; n += 2)
          pk[n / 2] = h2_as_u32(__floats2half2_rn(s[n] * (dp[n] - dl), s[n + 1] * (dp[n + 1] - dl)));
        if (!wait(&bar[R3_DS_EMPTY], (t & 1) ^ 1)) break;
#pragma unroll
        for (int x = 0; x < 4; ++x)
          sts_v4(sS_u + panel_off_u(128, row, col0 + 8 * x), pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[R3_DS_FULL]);
      }
      if (*s_abort) break;
    }

    // epilogue
    if (!C::ROWQ) {
      // merge the row's NCH chunk partials in chunk order
      if (C::NCH > 1) {
        if (ch > 0) {
          float* m = s_merge + ((ch - 1) * 128 + row) * 3;
          m[0] = m2, m[1] = l, m[2] = sd;
        }
        named_bar_sync(1, 32 * C::NSOFT);
      }
      if (ch == 0 && rvalid) {
        float mm = m2;
#pragma unroll
        for (int c = 1; c < C::NCH; ++c) mm = fmaxf(mm, s_merge[((c - 1) * 128 + row) * 3]);
        float L = 0.f, SD = 0.f;
        if (mm > -CUDART_INF_F) {
          const float fa = ex2(m2 - mm);
          L = l * fa, SD = sd * fa;
#pragma unroll
          for (int c = 1; c < C::NCH; ++c) {
            const float* m = s_merge + ((c - 1) * 128 + row) * 3;
            const float fb = ex2(m[0] - mm);
            L = fmaf(m[1], fb, L);
            SD = fmaf(m[2], fb, SD);
          }
        }
        float* o = p.part + (((size_t)split * p.Hkv + hk) * R + r) * 3;
        o[0] = mm, o[1] = L, o[2] = SD;
      }
    } else {
      // dQ; with key splits the scaled partial, completed by the split reduce
      float* out = !rvalid         ? nullptr
                   : p.nsplit > 1 ? p.dqpart + (((size_t)split * p.Hkv + hk) * R + r) * D
                                  : p.dQ + ((size_t)i * p.H + h) * D;
      const bool have = ntiles > 0 && wait(&bar[R3_ACC_FULL], 0);
      if (have) tc_fence_after();
#pragma unroll 1
      for (int c = col0; c < D; c += 32 * C::NCH) {
        float v[32];
        if (have) {
          tmem_ld32(tbase + C::T_ACC + lane_off + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= dq_fac;
        if (out) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(out + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (warp == 0 && lane == 0) {
      drain_loads(&bar[R3_K_FULL], C::KSTAGES, n_kload, deadline);
      drain_loads(&bar[R3_V_FULL], C::VSTAGES, n_vload, deadline);
      if (C::ROWQ && ntiles > 0) mbar_wait_until(&bar[R3_Q_FULL], 0, deadline);
      if (n_prod > 0) {
        mma_commit(&bar[R3_DRAIN0]);
        mbar_wait_until(&bar[R3_DRAIN0], 0, deadline);
      }
    }
    if ((warp == 1 || (C::DP_OWN && warp == C::W_DP)) && lane == 0 && s_issued) {
      uint64_t* dr = &bar[warp == 1 ? R3_DRAIN1 : R3_DRAIN2];
      mma_commit(dr);
      mbar_wait_until(dr, 0, deadline);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// Merge the split partials: lse and delta outputs plus the gradient passes' per-row values.
// With sink logits sigma_h, the sink joins the denominator as one more term e^sigma that has no
// value row: lse = log(e^sigma + sum_j e^s_j), and the keys' weights then sum to 1 - p_sink with
// p_sink = e^(sigma - lse).  delta = sum_j p_j dP_j is still the keys' sum, but the shift by r' no
// longer cancels in it: the shifted delta the gradient passes subtract is
//   delta - dO_i . r' = SD / L - p_sink dO_i . r'      (accumulator units: times sdO sV),
// and the row's term of the sink gradient is -p_sink delta (summed per head by k_sink_grad).
static __global__ void __launch_bounds__(256) k_lse_merge(Params p) {
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
  float sink2 = -CUDART_INF_F;  // the sink logit in log2 units
  if (p.sinks) {
    sink2 = p.sinks[h] * kLog2e;
    const float mm = fmaxf(m2, sink2);
    const float f = m2 > -CUDART_INF_F ? exp2f(m2 - mm) : 0.f;
    l = fmaf(l, f, exp2f(sink2 - mm));
    sd *= f;
    m2 = mm;
  }
  if (l > 0.f) {
    const float lse2 = m2 + log2f(l);
    const float ps = p.sinks ? exp2f(sink2 - lse2) : 0.f;
    const float dl = sd / l - ps * p.dOr[idx] * (st->sdO * st->sV);
    const float delta = dl * st->delta_fac + p.dOr[idx];
    p.lse2[idx] = lse2;
    p.dlt[idx] = dl;
    p.lse[(size_t)i * p.H + h] = lse2 * kLn2;
    if (p.delta) p.delta[(size_t)i * p.H + h] = delta;
    if (p.sg) p.sg[idx] = -ps * delta;
  } else {
    p.lse2[idx] = -CUDART_INF_F;
    p.dlt[idx] = 0.f;
    p.lse[(size_t)i * p.H + h] = -CUDART_INF_F;
    if (p.delta) p.delta[(size_t)i * p.H + h] = 0.f;
    if (p.sg) p.sg[idx] = 0.f;
  }
}

// Gradient of the sink logits: dsinks_h = sum_i -p_sink(i, h) delta_ih, the per-row terms of
// k_lse_merge summed in a fixed order (one block per head; thread t takes rows t, t + 256, ...
// in order, in double, then a fixed tree over the threads), so the result is deterministic.
static __global__ void __launch_bounds__(256) k_sink_grad(Params p) {
  __shared__ double part[256];
  const int h = blockIdx.x, hk = h / p.G, g = h % p.G;
  double acc = 0.0;
  for (int i = threadIdx.x; i < p.N; i += 256) acc += (double)p.sg[(size_t)hk * p.R + (size_t)i * p.G + g];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.dsinks[h] = (float)part[0];
}

// Fills the outputs of a problem without keys that has sink logits: every row's softmax holds the
// sink alone, so lse = sigma_h, delta = 0 and dQ = 0 (filled by the caller), and dsinks = 0.
static __global__ void k_sink_only(const float* sinks, float* lse, float* delta, float* dsinks, int N, int H) {
  const long idx = (long)blockIdx.x * 256 + threadIdx.x;
  if (idx < (long)N * H) {
    lse[idx] = sinks[idx % H];
    if (delta) delta[idx] = 0.f;
  }
  if (dsinks && idx < H) dsinks[idx] = 0.f;
}

// The per-row values of the gradient passes from a given lse and delta (instead of the LSE
// pass): lse2 = lse / ln 2 and the shifted delta in accumulator units, (delta - dO_i . r) sdO sV
// (the gradient passes take dP' - delta' with dP' = dO' . V', V' shifted by r).  A row whose lse
// is -inf (or not finite) has no allowed key.
static __global__ void __launch_bounds__(256) k_stats_in(Params p) {
  const long idx = (long)blockIdx.x * 256 + threadIdx.x;
  if (idx >= (long)p.Hkv * p.R) return;
  const int hk = (int)(idx / p.R), r = (int)(idx % p.R);
  const int i = r / p.G, h = hk * p.G + r % p.G;
  const float lse = p.lse_in[(size_t)i * p.H + h];
  if (!(lse > -CUDART_INF_F) || !isfinite(lse)) {
    p.lse2[idx] = -CUDART_INF_F;
    p.dlt[idx] = 0.f;
    return;
  }
  const Stats* st = p.st;
  p.lse2[idx] = lse * kLog2e;
  p.dlt[idx] = (p.delta_in[(size_t)i * p.H + h] - p.dOr[idx]) * (st->sdO * st->sV);
}

// dQ = sum of the split partials, in split order.
static __global__ void __launch_bounds__(256) k_dq_reduce(Params p) {
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
//
// A CTA owns BK keys of one KV head: their K' and V' tiles arrive once in shared memory (by TMA
// from the binary16 copies where the plan has them, else decoded here from the raw cache), then
// the CTA walks the 128-row query tiles that can see them.  Per query tile:
//   dP = dO V'^T, S = Q K'^T              (M = 128 rows, N = BK keys)
//   P                                     (softmax warps, written as binary16 [row][key])
//   dV^T += dO^T P, while the softmax forms dS = P * (dP - delta)
//   dK^T += Q^T dS                        (M = 128 feature rows per half, N = BK keys, K = 128 rows)
// Q and dO arrive as 64-column TMA panels with one full/empty barrier pair each; a panel is
// released when the last product reading it completes, so the next tile's loads overlap this
// tile's final products without a second buffer.
// Warp roles (12 warps): 0 producer, 1 MMA issuer / tensor-memory owner, 4-11 softmax and
// epilogue; without the binary16 copies every warp decodes K' and V' at the start.  Where the
// plan keeps dS for a separate dQ product (p.ds), the copy it stores is scaled by each row's own
// power of two (p.lamr) rather than the common multiplier of the dK^T operand: dQ is formed per
// row, so rows whose dO is much smaller than the largest keep binary16's relative precision.  The
// softmax writes that copy into the P panel once the dV^T product has read P, and warp 2 stores
// it with TMA; the next tile's P waits for the store to have read the panel.

template <int D, int Dv, int BK>
struct Cols2Cfg {
  static constexpr int NQP = D / 64, NOP = Dv / 64;  // panels of Q and dO
  static constexpr int KB = BK * D * 2, VB = BK * Dv * 2, QB = 128 * D * 2, OB = 128 * Dv * 2, PB = 128 * BK * 2;
  static constexpr int OFF_K = 0, OFF_V = KB, OFF_Q = KB + VB, OFF_O = OFF_Q + QB, OFF_P = OFF_O + OB,
                       OFF_S = OFF_P + PB, OFF_BAR = OFF_S + PB;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int NDH = D >= 128 ? D / 128 : 1, NVH = Dv >= 128 ? Dv / 128 : 1;
  static constexpr int T_S = 0, T_P = BK, T_V = 2 * BK, T_K = 2 * BK + NVH * BK;
  static constexpr int TCOLS = pow2_at_least(2 * BK + (NDH + NVH) * BK);
  static constexpr int HALF = BK / 2;
};

enum {
  C_Q_FULL = 0,   // [4]
  C_Q_EMPTY = 4,  // [4]
  C_O_FULL = 8,   // [4]
  C_O_EMPTY = 12, // [4]
  C_S_FULL = 16,
  C_P_FULL,   // the softmax wrote P (dV product may start)
  C_P_EMPTY,  // the dV product read P
  C_DS_FULL,
  C_DS_EMPTY,
  C_DONE,
  C_KV_FULL,   // K'/V' tiles loaded from the binary16 copies (levels 2 and 1)
  C_DSR_FULL,  // the softmax left this tile's per-row-scaled dS in the P panel (stored dS only)
  C_PS_EMPTY,  // the TMA store read that copy: the P panel may take the next tile's P
  C_COUNT
};
static_assert(8 * C_COUNT + 8 <= 256, "dK/dV pass barrier area");

// ROWCOPY selects the variant whose stored dS takes per-row multipliers.  Both variants are
// launched where dS is stored; each reads the decision (rows_need_own_scale, from the statistics
// on the device) first and returns at once unless it is the one that applies.  Separate variants
// keep the copy's code out of the common one: built into one kernel behind a run-time branch, it
// slowed the pass by about 5 % even where the branch was never taken.
template <int D, int Dv, int BK, bool ROWCOPY, bool EXT = false>
static __global__ void __launch_bounds__(384, 1)
    k_cols2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
            const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmKd,
            const __grid_constant__ CUtensorMap tmVd, Params p) {
  using C = Cols2Cfg<D, Dv, BK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sO = sm + C::OFF_O;
  uint8_t* sP = sm + C::OFF_P;
  uint8_t* sS = sm + C::OFF_S;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * C_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * C_COUNT + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kt = blockIdx.x, hk = blockIdx.y;
  const int j0 = kt * BK;
  const int R = p.R, G = p.G;
  int qt_begin = 0;
  if (p.causal) {
    const long imin = (long)j0 - ((long)p.M - p.N);  // first query that sees key j0
    if (imin > 0) qt_begin = (int)min((long)p.nQT, (imin * G) / 128);
  }
  const int nq = R > 0 ? max(0, p.nQT - qt_begin) : 0;

  // the dS kept for the dQ product: the dK^T operand's panel as it is, or a copy with each row's
  // own multiplier (left by the softmax in the P panel) when rows differ widely in size
  constexpr bool rowcopy = ROWCOPY;
  if (ROWCOPY != (p.ds != nullptr && rows_need_own_scale(*p.st))) return;  // the other variant applies
  if (warp == 1) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int c = 0; c < 4; ++c) {
      mbar_init(&bar[C_Q_FULL + c], 1);
      mbar_init(&bar[C_Q_EMPTY + c], 1);
      mbar_init(&bar[C_O_FULL + c], 1);
      mbar_init(&bar[C_O_EMPTY + c], 1);
    }
    mbar_init(&bar[C_S_FULL], 1);
    mbar_init(&bar[C_P_FULL], 8);
    mbar_init(&bar[C_P_EMPTY], 1);
    mbar_init(&bar[C_DS_FULL], 8);
    mbar_init(&bar[C_DS_EMPTY], (p.ds && !rowcopy) ? 2 : 1);  // the dK^T product (and the store)
    mbar_init(&bar[C_DONE], 1);
    mbar_init(&bar[C_KV_FULL], 1);
    mbar_init(&bar[C_DSR_FULL], 8);
    mbar_init(&bar[C_PS_EMPTY], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  const Stats st = *p.st;
  const bool kv_copies = p.kd != nullptr;  // K'/V' by TMA from the binary16 copies, else decoded here
  if (nq > 0 && !kv_copies) {  // K' and V' once, by every thread
    decode_tile<D, BK, 384>(p.k, p.k_type, p.rbk, hk, p.Hkv, j0, p.M, sK, st.sK, nullptr, tid);
    decode_tile<Dv, BK, 384>(p.v, p.v_type, p.rbv, hk, p.Hkv, j0, p.M, sV, st.sV, p.rsh + (size_t)hk * Dv, tid);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  int n_oload = 0, n_qload = 0;  // producer: dO and Q panels loaded

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmO);
      if (nq > 0 && kv_copies) {  // the key tile's K' and V' panels (same values as decode_tile's)
        mbar_arrive_expect_tx(&bar[C_KV_FULL], (uint32_t)(C::KB + C::VB));
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_3d(sK + c * BK * 128, &tmKd, &bar[C_KV_FULL], 0, j0, hk * (D / 64) + c);
#pragma unroll
        for (int c = 0; c < Dv / 64; ++c)
          tma_load_3d(sV + c * BK * 128, &tmVd, &bar[C_KV_FULL], 0, j0, hk * (Dv / 64) + c);
      }
      for (int t = 0; t < nq; ++t) {
        const int r0 = (qt_begin + t) * 128;
        // dO first: the dP product comes first, and the dV product frees its panels first
        bool ok = true;
        for (int c = 0; ok && c < C::NOP; ++c) {
          if (!(ok = wait(&bar[C_O_EMPTY + c], (t & 1) ^ 1))) break;
          mbar_arrive_expect_tx(&bar[C_O_FULL + c], 128 * 128);
          tma_load_3d(sO + c * 128 * 128, &tmO, &bar[C_O_FULL + c], c * 64, r0, hk);
          ++n_oload;
        }
        for (int c = 0; ok && c < C::NQP; ++c) {
          if (!(ok = wait(&bar[C_Q_EMPTY + c], (t & 1) ^ 1))) break;
          mbar_arrive_expect_tx(&bar[C_Q_FULL + c], 128 * 128);
          tma_load_3d(sQ + c * 128 * 128, &tmQ, &bar[C_Q_FULL + c], c * 64, r0, hk);
          ++n_qload;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && nq > 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
      constexpr uint32_t ID_T = idesc_f16(128, BK, true, true);
      constexpr uint32_t LBO_O = Dv >= 128 ? 128 * 128 : 0;  // second 64-row block of dO^T (repeat if Dv = 64)
      constexpr uint32_t LBO_Q = D >= 128 ? 128 * 128 : 0;
      const uint32_t tS = tbase + C::T_S, tP = tbase + C::T_P, tV = tbase + C::T_V, tK = tbase + C::T_K;
      // operand descriptors (K-major for S and dP; MN-major Q^T, dO^T and dS, P for the gradients)
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024), do0 = sdesc_sw128(smem_u32(sO), 16, 1024),
                     dk0 = sdesc_sw128(smem_u32(sK), 16, 1024), dv0 = sdesc_sw128(smem_u32(sV), 16, 1024),
                     dqt = sdesc_sw128(smem_u32(sQ), LBO_Q, 1024), dot = sdesc_sw128(smem_u32(sO), LBO_O, 1024),
                     ds0 = sdesc_sw128(smem_u32(sS), 128 * 128, 1024), dp0 = sdesc_sw128(smem_u32(sP), 128 * 128, 1024);
      const bool nq_ok = !kv_copies || wait(&bar[C_KV_FULL], 0);
      // Per query tile: dP, then S (so the Q panels, released last, have dP's time to arrive),
      // then dV^T once P is written and dK^T once dS is: the softmax's dS arithmetic overlaps
      // the dV^T product.
      for (int t = 0; nq_ok && t < nq; ++t) {
        bool ok = true;
        for (int c = 0; ok && c < C::NOP; ++c) {
          if (!(ok = wait(&bar[C_O_FULL + c], t & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16(tP, sdesc_adv(do0, c * (128 * 128) + k * 32), sdesc_adv(dv0, c * (BK * 128) + k * 32), ID_S,
                    (c > 0 || k > 0) ? 1u : 0u);
        }
        for (int c = 0; ok && c < C::NQP; ++c) {
          if (!(ok = wait(&bar[C_Q_FULL + c], t & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16(tS, sdesc_adv(dq0, c * (128 * 128) + k * 32), sdesc_adv(dk0, c * (BK * 128) + k * 32), ID_S,
                    (c > 0 || k > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(&bar[C_S_FULL]);
        const uint32_t acc0 = t > 0 ? 1u : 0u;
        if (!wait(&bar[C_P_FULL], t & 1)) break;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < C::NVH; ++hh) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16(tV + hh * BK, sdesc_adv(dot, hh * 2 * (128 * 128) + k * 2048), sdesc_adv(dp0, k * 2048), ID_T,
                    (acc0 || k > 0) ? 1u : 0u);
          mma_commit(&bar[C_O_EMPTY + 2 * hh]);
          if (2 * hh + 1 < C::NOP) mma_commit(&bar[C_O_EMPTY + 2 * hh + 1]);
        }
        mma_commit(&bar[C_P_EMPTY]);
        if (!wait(&bar[C_DS_FULL], t & 1)) break;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < C::NDH; ++hh) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16(tK + hh * BK, sdesc_adv(dqt, hh * 2 * (128 * 128) + k * 2048), sdesc_adv(ds0, k * 2048), ID_T,
                    (acc0 || k > 0) ? 1u : 0u);
          mma_commit(&bar[C_Q_EMPTY + 2 * hh]);
          if (2 * hh + 1 < C::NQP) mma_commit(&bar[C_Q_EMPTY + 2 * hh + 1]);
        }
        mma_commit(&bar[C_DS_EMPTY]);
      }
      mma_commit(&bar[C_DONE]);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ stored dS (dQ product)
    if (lane == 0 && p.ds) {
      prefetch_tmap(&tmS);
      for (int t = 0; t < nq; ++t) {
        if (!wait(&bar[rowcopy ? C_DSR_FULL : C_DS_FULL], t & 1)) break;
        uint8_t* src = rowcopy ? sP : sS;
#pragma unroll
        for (int c = 0; c < BK / 64; ++c)
          tma_store_3d(&tmS, src + c * (128 * 128), 0, 0, (hk * p.nQT + qt_begin + t) * p.ldds + j0 / 64 + c);
        bulk_commit_group();
        bulk_wait_read_all();  // the panel may be overwritten once read
        mbar_arrive(&bar[rowcopy ? C_PS_EMPTY : C_DS_EMPTY]);
      }
      bulk_wait_all();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax, then epilogue
    const int q4 = warp & 3, ch = (warp - 4) >> 2;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    auto row_stats = [&](int t, float& lse2, float& dl, float& lr, long& jlast, const uint16_t*& mrow) {
      const int r = (qt_begin + t) * 128 + row;
      const bool rvalid = r < R;
      const int i = rvalid ? r / G : 0;
      const int h = hk * G + (rvalid ? r % G : 0);
      lse2 = rvalid ? p.lse2[(size_t)hk * R + r] : -CUDART_INF_F;
      dl = rvalid ? p.dlt[(size_t)hk * R + r] : 0.f;
      lr = (rvalid && rowcopy) ? p.lamr[(size_t)hk * R + r] * (1.f / 32768.f) : 0.f;  // row multiplier / sP
      jlast = rvalid ? (p.causal ? min((long)p.M - 1, (long)p.M - p.N + i) : (long)p.M - 1) : -1;
      mrow = p.mask ? p.mask + ((size_t)(h % p.Hm) * p.N + i) * p.M : nullptr;
    };
    float lse2 = 0.f, dl = 0.f, lr = 0.f;
    float dls = 0.f;  // delta subtracted from dP in dS: the row's, or 0 where ext_scores has done it
    long jlast = -1;
    const uint16_t* mrow = nullptr;
    constexpr bool keep = ROWCOPY;
    // this thread's 32 values of the stored dS copy (row multiplier lr; 0 for a row past R)
    auto ds_row = [&](const float* pv, const float* dpv, uint32_t* w) {
#pragma unroll
      for (int x = 0; x < 32; x += 2)
        w[x / 2] = h2_as_u32(__floats2half2_rn(pv[x] * (dpv[x] - dls) * lr, pv[x + 1] * (dpv[x + 1] - dls) * lr));
    };
    // once the dV^T product of tile t has read P, the stored dS copy goes into the P panel
    auto put_ds_copy = [&](int t, int col0, const uint32_t* w, int nchunk) -> bool {
      if (!wait(&bar[C_P_EMPTY], t & 1)) return false;
      for (int c = 0; c < nchunk; ++c)
#pragma unroll
        for (int g = 0; g < 4; ++g)
          sts_v4(smem_u32(sP) + panel_off_u(128, row, col0 + 32 * c + 8 * g), w[16 * c + 4 * g], w[16 * c + 4 * g + 1],
                 w[16 * c + 4 * g + 2], w[16 * c + 4 * g + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[C_DSR_FULL]);
      return true;
    };
    const uint32_t sP_u = smem_u32(sP), sS_u = smem_u32(sS);
    // the exponent carries log2 of the P multiplier (a power of two), so the exponential is
    // the scaled P directly and dS takes lam / sP
    const float c2 = st.c2, lp = (float)ilogbf(st.sP), lam = st.lam / st.sP;
    if (nq > 0) row_stats(0, lse2, dl, lr, jlast, mrow);
    for (int t = 0; t < nq; ++t) {
      float nlse2 = 0.f, ndl = 0.f, nlr = 0.f;  // next tile's row values, fetched ahead
      long njlast = -1;
      const uint16_t* nmrow = nullptr;
      if (t + 1 < nq) row_stats(t + 1, nlse2, ndl, nlr, njlast, nmrow);
      const float nl = lse2 > -CUDART_INF_F ? lp - lse2 : -CUDART_INF_F;  // sP * p = 2^(t2 + nl); 0 on a dead row
      const int rcur = (qt_begin + t) * 128 + row;
      dls = EXT ? 0.f : dl;
      if (!wait(&bar[C_S_FULL], t & 1)) break;
      // the previous tile's P panel is free once its dV product (and the store of its dS copy) read it
      if (!wait(&bar[C_P_EMPTY], (t & 1) ^ 1)) break;
      if (keep && !wait(&bar[C_PS_EMPTY], (t & 1) ^ 1)) break;
      tc_fence_after();
      // log2-domain exponents of one 32-key chunk; a fully visible chunk without a mask takes
      // no per-key tests
      // (with the score extensions, dP also becomes (dP - delta) times the soft cap's derivative)
      auto exponents = [&](int col0, float* v, float* dpv) {
        if constexpr (EXT) {
          ext_scores<2>(v, dpv, j0 + col0, rcur, hk, nl, dl, jlast, mrow, st, p.alibi, G, p.M - p.N);
        } else if (mrow == nullptr && (long)(j0 + col0 + 31) <= jlast) {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = fmaf(v[x], c2, nl);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int j = j0 + col0 + x;
            bool ok = (long)j <= jlast;
            float mv = 0.f;
            if (ok && mrow) {
              mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
              ok = !(mv == -CUDART_INF_F);
            }
            v[x] = ok ? fmaf(v[x], c2, mv * kLog2e) + nl : -CUDART_INF_F;
          }
        }
      };
      if constexpr (C::HALF == 32) {
        // one chunk per thread: P is written and handed to the dV product first, then dS
        const int col0 = ch * 32;
        float s[32], dp[32];
        tmem_ld32(tbase + C::T_S + lane_off + col0, s);
        tmem_ld32(tbase + C::T_P + lane_off + col0, dp);
        tmem_ld_wait();
        exponents(col0, s, dp);
#pragma unroll
        for (int x = 0; x < 32; ++x) s[x] = ex2(s[x]);  // sP * p; 0 for masked keys and dead rows
#pragma unroll
        for (int g = 0; g < 32; g += 8)
          sts_v4(sP_u + panel_off_u(128, row, col0 + g), h2_as_u32(__floats2half2_rn(s[g], s[g + 1])),
                 h2_as_u32(__floats2half2_rn(s[g + 2], s[g + 3])), h2_as_u32(__floats2half2_rn(s[g + 4], s[g + 5])),
                 h2_as_u32(__floats2half2_rn(s[g + 6], s[g + 7])));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[C_P_FULL]);
        uint32_t pd[16], pr[16];
#pragma unroll
        for (int x = 0; x < 32; x += 2)
          pd[x / 2] = h2_as_u32(__floats2half2_rn(s[x] * (dp[x] - dls) * lam, s[x + 1] * (dp[x + 1] - dls) * lam));
        if (keep) ds_row(s, dp, pr);
        // the previous tile's dS panel is free once its dK product (and its store) read it
        if (!wait(&bar[C_DS_EMPTY], (t & 1) ^ 1)) break;
#pragma unroll
        for (int g = 0; g < 4; ++g)
          sts_v4(sS_u + panel_off_u(128, row, col0 + 8 * g), pd[4 * g], pd[4 * g + 1], pd[4 * g + 2], pd[4 * g + 3]);
        if (keep) {
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[C_DS_FULL]);
          if (!put_ds_copy(t, col0, pr, 1)) break;
        }
      } else {
        if (!wait(&bar[C_DS_EMPTY], (t & 1) ^ 1)) break;
        uint32_t pr[C::HALF / 2];
#pragma unroll
        for (int c = 0; c < C::HALF; c += 32) {
          const int col0 = ch * C::HALF + c;
          float s[32], dp[32];
          tmem_ld32(tbase + C::T_S + lane_off + col0, s);
          tmem_ld32(tbase + C::T_P + lane_off + col0, dp);
          tmem_ld_wait();
          exponents(col0, s, dp);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[x] = ex2(s[x]);  // sP * p; 0 for masked keys and dead rows
          if (keep) ds_row(s, dp, pr + c / 2);
#pragma unroll
          for (int g = 0; g < 32; g += 8) {
            uint32_t pp[4], pd[4];
#pragma unroll
            for (int n = 0; n < 8; n += 2) {
              const int x = g + n;
              const float p0 = s[x], p1 = s[x + 1];
              pp[n / 2] = h2_as_u32(__floats2half2_rn(p0, p1));
              pd[n / 2] = h2_as_u32(__floats2half2_rn(p0 * (dp[x] - dls) * lam, p1 * (dp[x + 1] - dls) * lam));
            }
            const uint32_t off = panel_off_u(128, row, col0 + g);
            sts_v4(sP_u + off, pp[0], pp[1], pp[2], pp[3]);
            sts_v4(sS_u + off, pd[0], pd[1], pd[2], pd[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[C_P_FULL]);
        if (keep) {
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[C_DS_FULL]);
          if (!put_ds_copy(t, ch * C::HALF, pr, C::HALF / 32)) break;
        }
      }
      if (*s_abort) break;
      if (!keep) {
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[C_DS_FULL]);
      }
      lse2 = nlse2, dl = ndl, lr = nlr, jlast = njlast, mrow = nmrow;
    }
    // epilogue: lane = feature row of a half, columns = keys; this warp takes half the keys
    const bool have = nq > 0 && wait(&bar[C_DONE], 0);
    if (have) tc_fence_after();
    const int lrow = q4 * 32 + lane;
#pragma unroll 1
    for (int hh = 0; hh < C::NVH + C::NDH; ++hh) {
      const bool isv = hh < C::NVH;
      const int half = isv ? hh : hh - C::NVH;
      const int DD = isv ? Dv : D;
      const int d = half * 128 + lrow;
      float* out = isv ? p.dV : p.dK;
      const float fac = isv ? st.dv_fac : st.dk_fac;
      const uint32_t tcol = isv ? C::T_V + half * BK : C::T_K + half * BK;
#pragma unroll 1
      for (int c = ch * C::HALF; c < (ch + 1) * C::HALF; c += 32) {
        float v[32];
        if (have) {
          tmem_ld32(tbase + tcol + lane_off + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (d < DD) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = j0 + c + e;
            if (j < p.M) out[((size_t)j * p.Hkv + hk) * DD + d] = v[e] * fac;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (warp == 0 && lane == 0) {
      if (nq > 0 && kv_copies) mbar_wait_until(&bar[C_KV_FULL], 0, deadline);
      drain_loads(&bar[C_O_FULL], C::NOP, n_oload, deadline);
      drain_loads(&bar[C_Q_FULL], C::NQP, n_qload, deadline);
    }
    // the issuer committed every product it issued to C_DONE before leaving its loop
    if (warp == 1 && lane == 0 && nq > 0) mbar_wait_until(&bar[C_DONE], 0, deadline);
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// Failure-detection self-test: one thread waits on an mbarrier nothing arrives on, gives up
// after limit_ns (the path every bounded wait of the backward takes) and records the timeout.
static __global__ void k_wait_selftest(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) record_error(err, kErrTimeout);
  }
}

// Fill kernel for degenerate shapes (a value into n floats).
static __global__ void k_fill(float* x, long n, float v) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < n) x[idx] = v;
}

// ------------------------------------------------------------------------------------------------
// dQ as one product over the stored dS: dQ_r = dq_fac * sum_j dS'_rj K'_j per (row tile, KV head,
// key split), over the key tiles the row tile can see.  dS' (binary16 lam * dS, written by the
// dK/dV pass) is the A operand (K-major, 64-key panels); K' is the B operand (MN-major).  Both
// arrive by TMA into a ring of stages; the accumulator is the whole 128 x D tile in tensor memory.
// Warp roles: 0 producer, 1 tensor-memory owner and MMA issuer, 4-7 epilogue.

template <int D, int BK>
struct GemmCfg {
  static constexpr int AB = 128 * BK * 2, BB = BK * D * 2, SB = AB + BB;  // bytes of one stage
  static constexpr int FIT = (232448 - 1024 - 256) / SB;
  static constexpr int NST = FIT < 6 ? FIT : 6;
  static constexpr int OFF_BAR = NST * SB;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + 1024 for aligning the base
  static constexpr int TCOLS = pow2_at_least(D);
  static_assert(NST >= 2 && SMEM <= 232448, "shared memory budget");
};

enum { G_FULL = 0, G_EMPTY = 6, G_ACC = 12, G_COUNT };

template <int D, int BK>
static __global__ void __launch_bounds__(256, 1)
    k_dq_gemm(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmK, Params p) {
  using C = GemmCfg<D, BK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * G_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * G_COUNT + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int r0 = qt * 128;
  const int R = p.R, G = p.G;
  const int kt_begin = split * p.kt_per_split;
  int kt_end = min(p.nKT, kt_begin + p.kt_per_split);
  if (p.causal) {
    const long i_hi = (long)min(R - 1, r0 + 127) / G;
    const long jmax = (long)p.M - p.N + i_hi;
    kt_end = min(kt_end, jmax < 0 ? 0 : (int)(jmax / BK) + 1);
  }
  const int ntiles = max(0, kt_end - kt_begin);

  if (warp == 1) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar[G_FULL + s], 1);
      mbar_init(&bar[G_EMPTY + s], 1);
    }
    mbar_init(&bar[G_ACC], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  int n_load = 0;  // producer: stages loaded

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmK);
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % C::NST;
        if (!wait(&bar[G_EMPTY + s], ((t / C::NST) & 1) ^ 1)) break;
        uint8_t* a = sm + s * C::SB;
        uint8_t* b = a + C::AB;
        const int j0 = (kt_begin + t) * BK;
        mbar_arrive_expect_tx(&bar[G_FULL + s], (uint32_t)C::SB);
#pragma unroll
        for (int c = 0; c < BK / 64; ++c)
          tma_load_3d(a + c * (128 * 128), &tmS, &bar[G_FULL + s], 0, 0, (hk * p.nQT + qt) * p.ldds + j0 / 64 + c);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(b + c * (BK * 128), &tmK, &bar[G_FULL + s], 0, j0, hk * (D / 64) + c);
        ++n_load;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID = idesc_f16(128, D, false, true);
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % C::NST;
        if (!wait(&bar[G_FULL + s], (t / C::NST) & 1)) break;
        tc_fence_after();
        const uint64_t da = sdesc_sw128(smem_u32(sm + s * C::SB), 16, 1024);
        const uint64_t db = sdesc_sw128(smem_u32(sm + s * C::SB + C::AB), BK * 128, 1024);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_f16(tbase, sdesc_adv(da, (k / 4) * (128 * 128) + (k % 4) * 32), sdesc_adv(db, k * 2048), ID,
                  (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bar[G_EMPTY + s]);
      }
      mma_commit(&bar[G_ACC]);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int r = r0 + row;
    const bool rvalid = r < R;
    const int i = rvalid ? r / G : 0;
    const int h = hk * G + (rvalid ? r % G : 0);
    float* out = !rvalid ? nullptr
                 : p.nsplit == 1 ? p.dQ + ((size_t)i * p.H + h) * D
                                 : p.dqpart + (((size_t)split * p.Hkv + hk) * R + r) * D;
    const Stats st = *p.st;
    const float dq_fac = !rvalid ? 0.f
                         : rows_need_own_scale(st) ? st.dq_fac * (st.lam / p.lamr[(size_t)hk * R + r])
                                                   : st.dq_fac;
    const bool have = ntiles > 0 && wait(&bar[G_ACC], 0);
    if (have) tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
      float v[32];
      if (have) {
        tmem_ld32(tbase + lane_off + c, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
      if (out) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(out + c + e) =
              make_float4(v[e] * dq_fac, v[e + 1] * dq_fac, v[e + 2] * dq_fac, v[e + 3] * dq_fac);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (warp == 0 && lane == 0) drain_loads(&bar[G_FULL], C::NST, n_load, deadline);
    // the issuer committed every product it issued to G_ACC before leaving its loop
    if (warp == 1 && lane == 0 && ntiles > 0) mbar_wait_until(&bar[G_ACC], 0, deadline);
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

}  // namespace fab
