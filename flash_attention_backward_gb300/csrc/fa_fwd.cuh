// Forward over the binary16 K'/V' copies in one pass: O and lse with an online softmax.
//
// A CTA owns 128 rows (r = i*G + g of one KV head) and the key tiles of one split, 64 keys per
// tile.  Per tile t:
//   S(t) = Q' K'(t)^T into one of two tensor-memory slots (Q' in tensor memory as the A operand,
//   K' from shared memory, K-major);
//   the softmax thread of each row takes its 64 scores, moves its running maximum m if needed,
//   writes P = 2^(s - m + kFwdLog2SP) as binary16 pairs over the first half of the same slot,
//   and adds their sum to l;
//   O += P(t) V'(t), with P as the tensor-memory A operand and V' as the MN-major B operand.
// The running maximum moves only when a score exceeds it by more than kFwdTau (log2 units);
// below that, P <= 2^(kFwdTau + kFwdLog2SP) = 2^15 stays inside binary16's range.  When it moves,
// every earlier product was taken against the old maximum: before it hands P(t) over, the row's
// thread waits for the product of tile t-1 to finish and multiplies its row of the accumulator by
// 2^(m_old - m_new) (a tensor-memory read and write of Dv columns; with the threshold it is rare
// after a row's first tiles).  Two threads issue the products: one the S products, the other
// the P V' products, each committing its own (a commit tracks only the committing thread's
// products).  An issuing thread is held while the pipe is busy and spends about as long again on
// its waits and commits; with two, one thread's bookkeeping runs while the other's products keep
// the pipe busy, and the S product of the next tile overlaps the P V' product of this one.
//
// With one split the epilogue writes O = acc / (sV l) + r' (V' holds v - r'; acc and l both in
// units of 2^kFwdLog2SP) and lse; with several, each split writes its unnormalised accumulator
// and (m, l), which k_fwd_merge combines in split order.
//
// Warp roles: 0 producer (TMA of K'/V' tiles into two rings), 1 tensor-memory owner and issuer of
// the S products, 2-5 softmax and epilogue (one per tensor-memory lane quarter: thread = row;
// they also write the rows of Q' into tensor memory), 6 issuer of the P V' products.
#pragma once
#include "fa_kernels.cuh"

namespace fab {

// P = 2^(s - m + kFwdLog2SP) with s - m <= kFwdTau (log2 units), so P <= 2^15
constexpr float kFwdLog2SP = 7.f, kFwdTau = 8.f, kFwdSP = 128.f;

template <int D, int Dv>
struct Fwd1Cfg {
  static constexpr int BK = 64;
  static constexpr int KB = BK * D * 2, VB = BK * Dv * 2;
  static constexpr int BAR_BYTES = 512;
  static constexpr int AVAIL = 232448 - 1024 - BAR_BYTES;
  // K'/V' stages (two to four each)
  static constexpr int NSTG = AVAIL / (KB + VB) >= 4 ? 4 : AVAIL / (KB + VB) >= 3 ? 3 : 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NSTG * KB;
  static constexpr int OFF_BAR = OFF_V + NSTG * VB;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + 1024 for aligning the base
  // tensor memory: [O accumulator: Dv columns] [S / P slot 0: BK] [S / P slot 1: BK] [Q': D / 2]
  static constexpr int T_O = 0, T_S = Dv, T_Q = Dv + 2 * BK;
  static constexpr int TCOLS = pow2_at_least(T_Q + D / 2);
  static constexpr int NT = 32 * 7;
  static_assert(NSTG * (KB + VB) <= AVAIL && SMEM <= 232448, "shared memory budget");
  static_assert(TCOLS <= 512, "tensor memory budget");
};

enum {
  F_K_FULL = 0,   // [4] K' tile landed
  F_K_EMPTY = 4,  // [4] its S product done
  F_V_FULL = 8,   // [4]
  F_V_EMPTY = 12, // [4] its P V' product done
  F_S_FULL = 16,  // [2] S(t) in slot t & 1
  F_P_FULL = 18,  // [2] P(t) written over slot t & 1 (and the accumulator rescaled), by the 4 softmax warps
  F_SLOT_FREE = 20,  // [2] the P V' product of the slot's last tile done: the slot may take S again
  F_PV_DONE = 22,    // one phase per P V' product
  F_O_FINAL,         // every P V' product done (the accumulator is final)
  F_Q_FULL,  // Q' in tensor memory (the 4 softmax warps)
  F_DRAIN,     // the S issuer's products, committed after an abort
  F_DRAIN_PV,  // the P V' issuer's products, committed after an abort
  F_COUNT
};
static_assert(8 * F_COUNT + 8 <= 512, "barrier area");

template <int D, int Dv>
static __global__ void __launch_bounds__(Fwd1Cfg<D, Dv>::NT, 1)
    k_fwd1(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Params p) {
  using C = Fwd1Cfg<D, Dv>;
  constexpr int BK = C::BK, NSTG = C::NSTG;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * F_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * F_COUNT + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int r0 = qt * 128;
  const int R = p.R, G = p.G;
  const int kt_begin = split * p.kt_per_split;  // in 64-key tiles
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
      mbar_init(&bar[F_K_FULL + s], 1);
      mbar_init(&bar[F_K_EMPTY + s], 1);
      mbar_init(&bar[F_V_FULL + s], 1);
      mbar_init(&bar[F_V_EMPTY + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[F_S_FULL + s], 1);
      mbar_init(&bar[F_P_FULL + s], 4);
      mbar_init(&bar[F_SLOT_FREE + s], 1);
    }
    mbar_init(&bar[F_PV_DONE], 1);
    mbar_init(&bar[F_O_FINAL], 1);
    mbar_init(&bar[F_Q_FULL], 4);
    mbar_init(&bar[F_DRAIN], 1);
    mbar_init(&bar[F_DRAIN_PV], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  const Stats st = *p.st;
  int n_k = 0, n_v = 0;  // producer: K' and V' tiles loaded
  bool issued = false;   // an issuer: any product issued

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      uint64_t t0 = globaltimer_ns();
      while (n_k < ntiles || n_v < ntiles) {
        bool moved = false;
        if (n_k < ntiles && mbar_try_wait(&bar[F_K_EMPTY + n_k % NSTG], ((n_k / NSTG) & 1) ^ 1)) {
          const int s = n_k % NSTG, j0 = (kt_begin + n_k) * BK;
          mbar_arrive_expect_tx(&bar[F_K_FULL + s], (uint32_t)C::KB);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sK + s * C::KB + c * (BK * 128), &tmK, &bar[F_K_FULL + s], 0, j0, hk * (D / 64) + c);
          ++n_k;
          moved = true;
        }
        if (n_v < ntiles && mbar_try_wait(&bar[F_V_EMPTY + n_v % NSTG], ((n_v / NSTG) & 1) ^ 1)) {
          const int s = n_v % NSTG, j0 = (kt_begin + n_v) * BK;
          mbar_arrive_expect_tx(&bar[F_V_FULL + s], (uint32_t)C::VB);
#pragma unroll
          for (int c = 0; c < Dv / 64; ++c)
            tma_load_3d(sV + s * C::VB + c * (BK * 128), &tmV, &bar[F_V_FULL + s], 0, j0, hk * (Dv / 64) + c);
          ++n_v;
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
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID_S = idesc_f16(128, BK, false, false);
      bool ok = wait(&bar[F_Q_FULL], 0);
      // S(t) into slot t & 1 once K'(t) has landed and the P V' product of the slot's last tile
      // (t - 2) is done
      for (int t = 0; ok && t < ntiles; ++t) {
        const int sl = t & 1, ks = t % NSTG;
        if (!wait(&bar[F_K_FULL + ks], (t / NSTG) & 1) || !wait(&bar[F_SLOT_FREE + sl], ((t >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        issued = true;
        tc_fence_after();
        const uint64_t dk = sdesc_sw128(smem_u32(sK + ks * C::KB), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_f16_tmem_a(tbase + C::T_S + sl * BK, tbase + C::T_Q + k * 8,
                         sdesc_adv(dk, (k / 4) * (BK * 128) + (k % 4) * 32), ID_S, k > 0);
        mma_commit(&bar[F_S_FULL + sl]);
        mma_commit(&bar[F_K_EMPTY + ks]);
      }
      if (issued) mma_commit(&bar[F_DRAIN]);  // every product issued above (also after an abort)
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------------ P V' issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID_O = idesc_f16(128, Dv, false, true);
      bool ok = true;
      // O += P(u) V'(u): P from its slot (binary16 pairs over the first BK / 2 columns)
      for (int u = 0; ok && u < ntiles; ++u) {
        const int sl = u & 1, vs = u % NSTG;
        if (!wait(&bar[F_P_FULL + sl], (u >> 1) & 1) || !wait(&bar[F_V_FULL + vs], (u / NSTG) & 1)) {
          ok = false;
          break;
        }
        issued = true;
        tc_fence_after();
        const uint64_t dv = sdesc_sw128(smem_u32(sV + vs * C::VB), BK * 128, 1024);
        const uint32_t ta = tbase + C::T_S + sl * BK;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_f16_tmem_a(tbase + C::T_O, ta + k * 8, sdesc_adv(dv, k * 2048), ID_O, (u > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bar[F_V_EMPTY + vs]);
        mma_commit(&bar[F_SLOT_FREE + sl]);
        mma_commit(&bar[F_PV_DONE]);
      }
      if (ok) mma_commit(&bar[F_O_FINAL]);
      if (issued) mma_commit(&bar[F_DRAIN_PV]);
    }
  } else {
    // ------------------------------------------------------------------ softmax, then epilogue
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int r = r0 + row;
    const bool rvalid = r < R;
    const int i = rvalid ? r / G : 0;
    const int h = hk * G + (rvalid ? r % G : 0);
    const long jlast = rvalid ? (p.causal ? min((long)p.M - 1, (long)p.M - p.N + i) : (long)p.M - 1) : -1;
    const uint16_t* mrow = p.mask ? p.mask + ((size_t)(h % p.Hm) * p.N + i) * p.M : nullptr;
    const float c2 = st.c2;
    // running maximum (log2 units), compensated sum of P (units of 2^kFwdLog2SP)
    float m = -CUDART_INF_F, l = 0.f, lc = 0.f;

    if (ntiles > 0) {
      // this row of Q' into tensor memory (binary16 pairs per column), the A operand of S
      const uint4* src = reinterpret_cast<const uint4*>(p.q16 + ((size_t)hk * R + (rvalid ? r : 0)) * D);
#pragma unroll 1
      for (int c = 0; c < D / 2; c += 32) {
        uint32_t wv[32];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const uint4 u = rvalid ? __ldg(src + c / 4 + x) : make_uint4(0, 0, 0, 0);
          wv[4 * x] = u.x, wv[4 * x + 1] = u.y, wv[4 * x + 2] = u.z, wv[4 * x + 3] = u.w;
        }
        tmem_st32(tbase + lane_off + C::T_Q + c, wv);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[F_Q_FULL]);
    }

    for (int t = 0; t < ntiles; ++t) {
      const int sl = t & 1;
      const int j0 = (kt_begin + t) * BK;
      const uint32_t tS = tbase + C::T_S + sl * BK + lane_off;
      if (!wait(&bar[F_S_FULL + sl], (t >> 1) & 1)) break;
      tc_fence_after();
      float x[2][32];
      tmem_ld32(tS, x[0]);
      tmem_ld32(tS + 32, x[1]);
      tmem_ld_wait();
      // log2-domain scores; masked keys -> -inf
      float mx[8];  // partial maxima (independent chains)
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int k0 = j0 + 32 * c;
        if (mrow == nullptr && (long)(k0 + 31) <= jlast) {
#pragma unroll
          for (int n = 0; n < 32; ++n) x[c][n] *= c2;
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            const int j = k0 + n;
            bool okj = (long)j <= jlast;
            float mv = 0.f;
            if (okj && mrow) {
              mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
              okj = !(mv == -CUDART_INF_F);
            }
            x[c][n] = okj ? fmaf(x[c][n], c2, mv * kLog2e) : -CUDART_INF_F;
          }
        }
#pragma unroll
        for (int n = 0; n < 32; ++n) mx[n & 7] = fmaxf(mx[n & 7], x[c][n]);
      }
      const float cmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // a maximum more than kFwdTau above the running one rescales what was summed (and, below,
      // accumulated) against the old one; the first live tile only sets it
      const bool grow = m > -CUDART_INF_F && cmax > m + kFwdTau;
      const float f = grow ? ex2(m - cmax) : 1.f;
      if (grow) {
        l *= f, lc *= f;
        m = cmax;
      } else if (m == -CUDART_INF_F) {
        m = cmax;
      }
      uint32_t pk[32];
      float cl = 0.f;
      if (m > -CUDART_INF_F) {
        const float mP = m - kFwdLog2SP;  // 2^(s - mP) = P
        float ca[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int n = 0; n < 32; n += 2) {
            const float e0 = ex2(x[c][n] - mP), e1 = ex2(x[c][n + 1] - mP);  // 0 for masked keys
            ca[(n >> 1) & 3] += e0 + e1;
            pk[16 * c + n / 2] = h2_as_u32(__floats2half2_rn(e0, e1));
          }
        cl = (ca[0] + ca[1]) + (ca[2] + ca[3]);
      } else {
#pragma unroll
        for (int n = 0; n < 32; ++n) pk[n] = 0u;
      }
      {  // compensated accumulation of the tile sums
        const float y = cl - lc, tt = l + y;
        lc = (tt - l) - y, l = tt;
      }
      tmem_st32(tS, pk);  // P over the first BK / 2 columns of the slot
      if (__any_sync(0xffffffffu, grow)) {
        // the accumulator holds the products of tiles < t: wait for the last, then rescale the
        // rows whose maximum grew (the others by 1)
        if (!wait(&bar[F_PV_DONE], (t - 1) & 1)) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < Dv; c += 32) {
          float o[32];
          tmem_ld32(tbase + C::T_O + lane_off + c, o);
          tmem_ld_wait();
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(o[e] * f);
          tmem_st32(tbase + C::T_O + lane_off + c, w);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[F_P_FULL + sl]);
      if (*s_abort) break;
    }

    // epilogue: one split writes O and lse; several write the unnormalised accumulator and
    // (m, l) for k_fwd_merge
    const bool have = ntiles > 0 && wait(&bar[F_O_FINAL], 0);
    if (have) tc_fence_after();
    const bool live = have && m > -CUDART_INF_F && l > 0.f;
    l *= 1.f / kFwdSP;  // exact: a power of two
    const float acc_fac = 1.f / (kFwdSP * st.sV);
    const bool whole = p.nsplit == 1;
    float* out = !rvalid ? nullptr
                 : whole ? p.o_out + ((size_t)i * p.H + h) * Dv
                         : p.dqpart + (((size_t)split * p.Hkv + hk) * R + r) * Dv;
    const float ofac = whole ? (live ? acc_fac / l : 0.f) : (live ? acc_fac : 0.f);
    const float* rsh = whole ? p.rmean + (size_t)hk * Dv : nullptr;
#pragma unroll 1
    for (int c = 0; c < Dv; c += 32) {
      float v[32];
      if (have) {
        tmem_ld32(tbase + C::T_O + lane_off + c, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = live ? v[e] * ofac + (rsh ? rsh[c + e] : 0.f) : 0.f;
      if (out) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(out + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
    if (rvalid) {
      if (whole) {
        p.lse[(size_t)i * p.H + h] = live ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
      } else {
        float* o = p.part + (((size_t)split * p.Hkv + hk) * R + r) * 3;
        o[0] = live ? m : -CUDART_INF_F, o[1] = live ? l : 0.f, o[2] = 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (warp == 0 && lane == 0) {
      drain_loads(&bar[F_K_FULL], NSTG, n_k, deadline);
      drain_loads(&bar[F_V_FULL], NSTG, n_v, deadline);
    }
    if (warp == 1 && lane == 0 && issued) mbar_wait_until(&bar[F_DRAIN], 0, deadline);
    if (warp == 6 && lane == 0 && issued) mbar_wait_until(&bar[F_DRAIN_PV], 0, deadline);
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// The forward's split partials combined per row, in split order: M = max m_s, L = sum l_s 2^(m_s - M),
// O = sum_s O_s 2^(m_s - M) / L + r' and lse = (M + log2 L) ln 2; a row without keys gets O = 0
// and lse = -inf.
static __global__ void __launch_bounds__(256) k_fwd_merge(Params p) {
  const long nv = (long)p.Hkv * p.R * (p.Dv / 4);
  const long idx = (long)blockIdx.x * 256 + threadIdx.x;
  if (idx >= nv) return;
  const long row = idx / (p.Dv / 4);
  const int c = (int)(idx % (p.Dv / 4)) * 4;
  const int hk = (int)(row / p.R), r = (int)(row % p.R);
  const int i = r / p.G, h = hk * p.G + r % p.G;
  float mm = -CUDART_INF_F;
  for (int s = 0; s < p.nsplit; ++s) mm = fmaxf(mm, p.part[(((size_t)s * p.Hkv + hk) * p.R + r) * 3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (mm > -CUDART_INF_F) {
    for (int s = 0; s < p.nsplit; ++s) {
      const float* q = p.part + (((size_t)s * p.Hkv + hk) * p.R + r) * 3;
      if (q[0] == -CUDART_INF_F) continue;
      const float f = exp2f(q[0] - mm);
      L = fmaf(q[1], f, L);
      const float4 x = *reinterpret_cast<const float4*>(p.dqpart + (((size_t)s * p.Hkv + hk) * p.R + r) * p.Dv + c);
      acc.x = fmaf(x.x, f, acc.x), acc.y = fmaf(x.y, f, acc.y), acc.z = fmaf(x.z, f, acc.z), acc.w = fmaf(x.w, f, acc.w);
    }
  }
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (L > 0.f) {
    const float inv = 1.f / L;
    const float* rm = p.rmean + (size_t)hk * p.Dv + c;
    o = make_float4(acc.x * inv + rm[0], acc.y * inv + rm[1], acc.z * inv + rm[2], acc.w * inv + rm[3]);
  }
  *reinterpret_cast<float4*>(p.o_out + ((size_t)i * p.H + h) * p.Dv + c) = o;
  if (c == 0) p.lse[(size_t)i * p.H + h] = L > 0.f ? (mm + log2f(L)) * kLn2 : -CUDART_INF_F;
}

}  // namespace fab
