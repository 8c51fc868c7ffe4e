// LSE/D pass on a pair of SMs, straight from the raw cache.
//
// Per row i of a query head the pass forms the statistics that define lse and D ("CUDA:
// FLASH_ATTN_BACK kernels", revision 8798492, the fused LSE/D pass): the running maximum m of
// s_ij, l = sum_j e^(s_ij - m) and sd = sum_j e^(s_ij - m) dP_ij, rescaled together when m grows,
// with lse = m + log l and D = sd / l.  S = Q' K'^T and dP = dO' V'^T are tensor-core products.
//
// A cluster of two CTAs owns two 128-row tiles (rows r = i*G + g of one KV head) and walks the
// key tiles of one split, 128 keys per tile.  The products run as cta_group::2 MMAs (M = 256):
//   * each CTA keeps its own rows' Q' and dO' in tensor memory (the A operands) and receives its
//     own rows of S and dP there;
//   * the B operand (K' or V' of the 128 keys) is split between the CTAs by keys: each CTA loads
//     the raw cache rows of its 64 keys by TMA and decodes them once into binary16 in its shared
//     memory ("masking and q8_0" review: each K/V element decoded once per tile, in pairs), and
//     the two halves meet in the tensor cores;
//   * one thread of the even CTA issues every product and commits it to both CTAs' barriers; the
//     odd CTA's decoders and softmax warps report to the even CTA by remote mbarrier arrives.
// So each SM decodes half of each tile and holds half of its operand in shared memory, and no
// binary16 copy of the cache is made.  The decoders round as k_predecode and decode_tile do, so
// every pass forms S and dP from identical operands.
//
// Warp roles per CTA: 0 producer (TMA of raw rows into a K ring and a V ring), 1 tensor-memory
// owner (collective allocation) and, in the even CTA, MMA issuer, 4-11 softmax (thread = row and
// half of the tile's keys), 2-3 and 12-19 decoders.  The decode runs on latency (about 0.6
// instructions per clock over six decoder warps), so it takes ten; the registers that allows come
// from a split per warpgroup: warpgroups 1 and 2 (softmax) take REG_SOFT each, warpgroups 0, 3
// and 4 (producer, issuer, decoders) REG_REST.  Every wait is bounded; neither CTA leaves before
// the other (cluster barrier) or before the products and arrivals aimed at it have landed.
#pragma once
#include "fa_kernels.cuh"

namespace fab {

// Bounded waits on barriers that the other CTA of the pair arrives on (acquire at cluster scope).
// A thread suspended in try_wait was measured to resume about a microsecond after a remote arrival
// completed the phase, so the MMA issuer, alone in its warp and on the critical path, polls with
// test_wait (Poll = true); the other roles sleep in try_wait and leave the issue slots to the
// decoders.
template <bool Poll>
struct WaiterC {
  volatile int* abort;
  int* err;
  uint64_t limit_ns;
  __device__ __forceinline__ bool test(uint64_t* bar, uint32_t parity) const {
    return Poll ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity);
  }
  __device__ __forceinline__ bool operator()(uint64_t* bar, uint32_t parity) const {
    if (test(bar, parity)) return true;
    if (*abort) return false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (test(bar, parity)) return true;
      if (((it & 255u) == 0 || limit_ns < kShortWaitNs) && globaltimer_ns() - t0 > limit_ns) break;
    }
    *abort = 1;
    record_error(err, kErrTimeout);
    return false;
  }
};

template <int D, int Dv>
struct LsePairCfg {
  static constexpr int BK = 128;     // keys per tile
  static constexpr int HK = BK / 2;  // keys decoded by each CTA
  static constexpr int KB = HK * D * 2, VB = HK * Dv * 2;
  static constexpr int STAGES = 2;
  static constexpr int NSOFT = 8, NCH = 2;  // softmax warps; key halves per row
  static constexpr int W_SOFT = 4, W_DEC = W_SOFT + NSOFT;  // first softmax warp; first decoder after them
  static constexpr int NDEC = 10;                           // decoder warps: 2, 3 and W_DEC ..
  static constexpr int NT = 32 * (W_DEC + NDEC - 2);
  static constexpr int REG_SOFT = 128, REG_REST = 72;       // registers per thread after the split
  static constexpr long REG_NEED = 128L * (2 * REG_SOFT + (NT / 128 - 2) * REG_REST);
  static_assert(NT % 128 == 0 && W_SOFT % 4 == 0 && NSOFT == 8, "roles on warpgroup boundaries");
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * KB;
  static constexpr int OFF_BAR = OFF_V + STAGES * VB;
  static constexpr int BAR_BYTES = 512 + (NCH - 1) * 128 * 3 * 4;  // barriers, then the row merge area
  static constexpr int OFF_RAW = OFF_BAR + BAR_BYTES;
  static constexpr int SMEM_MAX = 232448;
  static constexpr int RAW_BUDGET = SMEM_MAX - 1024 - 64 - OFF_RAW;  // bytes for the raw rings
  static constexpr int T_Q = 0, T_O = D / 2, T_S = T_O + Dv / 2, T_P = T_S + BK;
  static constexpr int TCOLS = pow2_at_least(T_P + BK);
  static_assert(TCOLS <= 512, "tensor memory budget");
  static_assert(RAW_BUDGET > 0, "shared memory budget");
};

enum {
  L_RK_FULL = 0,                        // [kMaxRawDepth] raw K entry landed
  L_RK_EMPTY = L_RK_FULL + kMaxRawDepth,  // [kMaxRawDepth] raw K entry decoded
  L_RV_FULL = L_RK_EMPTY + kMaxRawDepth,
  L_RV_EMPTY = L_RV_FULL + kMaxRawDepth,
  L_K_FULL = L_RV_EMPTY + kMaxRawDepth,  // [2] (even CTA) K' stage decoded in both CTAs
  L_V_FULL = L_K_FULL + 2,               // [2]
  L_K_EMPTY = L_V_FULL + 2,              // [2] (both) S product read the K' stage
  L_V_EMPTY = L_K_EMPTY + 2,             // [2]
  L_S_FULL = L_V_EMPTY + 2,              // (both) S in tensor memory
  L_P_FULL,                              // (both) dP in tensor memory
  L_S_FREE,                              // (even CTA) both CTAs' softmax read S
  L_P_FREE,                              // (even CTA) both CTAs' softmax read dP
  L_OPS_READY,                           // (even CTA) Q' and dO' in both CTAs' tensor memory
  L_DRAIN,                               // the issuer's products, committed after the last one
  L_COUNT
};
static_assert(8 * L_COUNT + 8 <= 512, "barrier area");

template <int D, int Dv, bool EXT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(LsePairCfg<D, Dv>::NT, 1)
    k_lse_pair(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Params p) {
  using C = LsePairCfg<D, Dv>;
  constexpr int BK = C::BK, HK = C::HK;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sRaw = sm + C::OFF_RAW;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * L_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * L_COUNT + 4);
  float* s_merge = reinterpret_cast<float*>(sm + C::OFF_BAR + 512);  // [128][3]

  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x >> 1, hk = blockIdx.y, split = blockIdx.z;
  const int r0 = (2 * pair + (int)rank) * 128;  // this CTA's rows
  const int R = p.R, G = p.G;
  // both CTAs walk the same key tiles: the causal bound of the pair's last row
  const int kt_begin = split * p.kt_per_split;
  int kt_end = min(p.nKT, kt_begin + p.kt_per_split);
  if (p.causal) {
    const long i_hi = (long)min(R - 1, (2 * pair + 1) * 128 + 127) / G;
    const long jmax = (long)p.M - p.N + i_hi;
    kt_end = min(kt_end, jmax < 0 ? 0 : (int)(jmax / BK) + 1);
  }
  const int ntiles = max(0, kt_end - kt_begin);
  const int KE = p.ke, EPT = HK / KE, RK = p.raw_depth, RV = p.raw_depth_v;
  const int kent = KE * p.rbk_pad, vent = KE * p.rbv_pad;  // bytes of one K / V ring entry
  uint8_t* sRawV = sRaw + RK * kent;

  if (warp == 1) tmem_alloc_pair(tslot, C::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < kMaxRawDepth; ++s) {
      mbar_init(&bar[L_RK_FULL + s], 1);
      mbar_init(&bar[L_RK_EMPTY + s], C::NDEC);
      mbar_init(&bar[L_RV_FULL + s], 1);
      mbar_init(&bar[L_RV_EMPTY + s], C::NDEC);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[L_K_FULL + s], 2 * C::NDEC);
      mbar_init(&bar[L_V_FULL + s], 2 * C::NDEC);
      mbar_init(&bar[L_K_EMPTY + s], 1);
      mbar_init(&bar[L_V_EMPTY + s], 1);
    }
    mbar_init(&bar[L_S_FULL], 1);
    mbar_init(&bar[L_P_FULL], 1);
    mbar_init(&bar[L_S_FREE], 2 * C::NSOFT);
    mbar_init(&bar[L_P_FREE], 2 * C::NSOFT);
    mbar_init(&bar[L_OPS_READY], 2 * C::NSOFT);
    mbar_init(&bar[L_DRAIN], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  // both CTAs' barriers and tensor memory exist before either CTA signals the other
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  const WaiterC<false> wait_c{s_abort, p.err, p.wait_ns};
  const WaiterC<true> poll_c{s_abort, p.err, p.wait_ns};
  const Stats st = *p.st;
  // the even CTA's barrier at the offset of local barrier `b`
  auto lead_bar = [&](int b) { return mapa_shared(smem_u32(&bar[b]), 0); };
  auto arrive_lead = [&](int b) {
    if (lead)
      mbar_arrive(&bar[b]);
    else
      mbar_arrive_remote(lead_bar(b));
  };
  int n_kraw = 0, n_vraw = 0;  // producer: raw entries loaded
  bool issued = false;         // issuer: any product issued

  // the register split, uniform within each warpgroup: each share governs the code it heads
  if (warp >= C::W_SOFT && warp < C::W_DEC) {
    setmaxnreg_inc<C::REG_SOFT>();
    // ------------------------------------------------------------------ softmax
    const int q4 = warp & 3, ch = (warp - C::W_SOFT) >> 2;  // tensor-memory lane quarter; half of the keys
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int col0 = ch * (BK / 2);
    const int r = r0 + row;
    const bool rvalid = r < R;
    const int i = rvalid ? r / G : 0;
    const int h = hk * G + (rvalid ? r % G : 0);
    const long jlast = rvalid ? (p.causal ? min((long)p.M - 1, (long)p.M - p.N + i) : (long)p.M - 1) : -1;
    const uint16_t* mrow = p.mask ? p.mask + ((size_t)(h % p.Hm) * p.N + i) * p.M : nullptr;
    const float c2 = st.c2;
    float m2 = -CUDART_INF_F, l = 0.f, lc = 0.f, sd = 0.f, sdc = 0.f;

    if (ntiles > 0) {
      // this thread's half of the row's A operands into tensor memory (binary16 pairs per column)
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
      put_row(p.q16 + rowq * D, D, C::T_Q);
      put_row(p.do16 + rowq * Dv, Dv, C::T_O);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_lead(L_OPS_READY);
    }

    for (int t = 0; t < ntiles; ++t) {
      const int j0 = (kt_begin + t) * BK;
      float e[2][32];
      if (!wait_c(&bar[L_S_FULL], t & 1)) break;
      tc_fence_after();
      tmem_ld32(tbase + C::T_S + lane_off + col0, e[0]);
      tmem_ld32(tbase + C::T_S + lane_off + col0 + 32, e[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_lead(L_S_FREE);
      // log2-domain scores of this thread's two 32-key chunks; masked keys -> -inf
      float cmax = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int k0 = j0 + col0 + 32 * c;
        if constexpr (EXT) {
          ext_scores<0>(e[c], nullptr, k0, r, hk, 0.f, 0.f, jlast, mrow, st, p.alibi, G, p.M - p.N);
        } else if (mrow == nullptr && (long)(k0 + 31) <= jlast) {
#pragma unroll
          for (int n = 0; n < 32; ++n) e[c][n] = e[c][n] * c2;
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            const int j = k0 + n;
            bool ok = (long)j <= jlast;
            float mv = 0.f;
            if (ok && mrow) {
              mv = h2f(__ldg(reinterpret_cast<const unsigned short*>(mrow) + j));
              ok = !(mv == -CUDART_INF_F);
            }
            e[c][n] = ok ? fmaf(e[c][n], c2, mv * kLog2e) : -CUDART_INF_F;
          }
        }
#pragma unroll
        for (int n = 0; n < 32; ++n) cmax = fmaxf(cmax, e[c][n]);
      }
      if (cmax > m2) {
        const float f = ex2(m2 - cmax);  // 0 while m2 = -inf
        l *= f, lc *= f, sd *= f, sdc *= f;
        m2 = cmax;
      }
      const bool any = cmax > -CUDART_INF_F;
      if (any) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int n = 0; n < 32; ++n) e[c][n] = ex2(e[c][n] - m2);
      }
      if (!wait_c(&bar[L_P_FULL], t & 1)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float dp[32];
        tmem_ld32(tbase + C::T_P + lane_off + col0 + 32 * c, dp);
        tmem_ld_wait();
        if (c == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_lead(L_P_FREE);
        }
        if (any) {
          float cl = 0.f, cs = 0.f;
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            cl += e[c][n];
            cs = fmaf(e[c][n], dp[n], cs);
          }
          // compensated accumulation of the chunk sums
          float y = cl - lc, tt = l + y;
          lc = (tt - l) - y, l = tt;
          y = cs - sdc, tt = sd + y;
          sdc = (tt - sd) - y, sd = tt;
        }
      }
      if (*s_abort) break;
    }
    // merge the row's two key halves in half order
    if (ch == 1) s_merge[row * 3 + 0] = m2, s_merge[row * 3 + 1] = l, s_merge[row * 3 + 2] = sd;
    named_bar_sync(1, 32 * C::NSOFT);
    if (ch == 0 && rvalid) {
      const float m2b = s_merge[row * 3 + 0], lb = s_merge[row * 3 + 1], sdb = s_merge[row * 3 + 2];
      const float mm = fmaxf(m2, m2b);
      float L = 0.f, SD = 0.f;
      if (mm > -CUDART_INF_F) {
        const float fa = ex2(m2 - mm), fb = ex2(m2b - mm);
        L = fmaf(lb, fb, l * fa);
        SD = fmaf(sdb, fb, sd * fa);
      }
      float* o = p.part + (((size_t)split * p.Hkv + hk) * R + r) * 3;
      o[0] = mm, o[1] = L, o[2] = SD;
    }
  } else {
    setmaxnreg_dec<C::REG_REST>();
    if (warp == 0) {
      // ------------------------------------------------------------------ producer
      if (lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        const int tot = ntiles * EPT;
        int ek = 0, ev = 0, sk = 0, uk = 0, sv = 0, uv = 0;
        uint64_t t0 = globaltimer_ns();
        // entry e of a ring holds keys e*KE.. of this CTA's halves of the split's tiles
        auto load_entry = [&](bool isv, int e, int slot) {
          const int t = e / EPT, h = e % EPT;
          const int ja = (kt_begin + t) * BK + (int)rank * HK + h * KE;
          const int nv = max(0, min(KE, p.M - ja));
          uint64_t* fb = &bar[(isv ? L_RV_FULL : L_RK_FULL) + slot];
          if (nv > 0) {
            mbar_arrive_expect_tx(fb, (uint32_t)(KE * (isv ? p.rbv : p.rbk)));
            tma_load_3d(isv ? sRawV + slot * vent : sRaw + slot * kent, isv ? &tmV : &tmK, fb, 0, hk, ja);
          } else {
            mbar_arrive(fb);
          }
        };
        while (ek < tot || ev < tot) {
          bool moved = false;
          if (ek < tot && mbar_try_wait(&bar[L_RK_EMPTY + sk], (uk & 1) ^ 1)) {
            load_entry(false, ek++, sk);
            if (++sk == RK) sk = 0, ++uk;
            moved = true;
          }
          if (ev < tot && mbar_try_wait(&bar[L_RV_EMPTY + sv], (uv & 1) ^ 1)) {
            load_entry(true, ev++, sv);
            if (++sv == RV) sv = 0, ++uv;
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
        n_kraw = ek, n_vraw = ev;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------ MMA issuer (even CTA)
      if (lead && lane == 0 && ntiles > 0) {
        constexpr uint32_t ID = idesc_f16(256, BK, false, false);
        const uint32_t tQ = tbase + C::T_Q, tO = tbase + C::T_O, tS = tbase + C::T_S, tP = tbase + C::T_P;
        if (poll_c(&bar[L_OPS_READY], 0)) {
          for (int t = 0; t < ntiles; ++t) {
            const int s = t & 1;
            if (!poll_c(&bar[L_K_FULL + s], (t >> 1) & 1) || !poll_c(&bar[L_S_FREE], (t & 1) ^ 1)) break;
            issued = true;
            tc_fence_after();
            const uint64_t db = sdesc_sw128(smem_u32(sK + s * C::KB), 16, 1024);
  #pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_f16_tmem_a_pair(tS, tQ + k * 8, sdesc_adv(db, (k / 4) * (HK * 128) + (k % 4) * 32), ID, k > 0);
            mma_commit_pair(&bar[L_S_FULL], 3);
            mma_commit_pair(&bar[L_K_EMPTY + s], 3);
            if (!poll_c(&bar[L_V_FULL + s], (t >> 1) & 1) || !poll_c(&bar[L_P_FREE], (t & 1) ^ 1)) break;
            tc_fence_after();
            const uint64_t dv = sdesc_sw128(smem_u32(sV + s * C::VB), 16, 1024);
  #pragma unroll
            for (int k = 0; k < Dv / 16; ++k)
              mma_f16_tmem_a_pair(tP, tO + k * 8, sdesc_adv(dv, (k / 4) * (HK * 128) + (k % 4) * 32), ID, k > 0);
            mma_commit_pair(&bar[L_P_FULL], 3);
            mma_commit_pair(&bar[L_V_EMPTY + s], 3);
          }
        }
        if (issued) mma_commit_pair(&bar[L_DRAIN], 1);  // every product above has completed
      }
    } else {
      // ------------------------------------------------------------------ decoders
      constexpr int NDT = C::NDEC * 32;
      static_assert(NDT % 64 == 0, "decoder_map needs a multiple of 8 column groups of 8 lanes");
      const int dt = (warp < C::W_SOFT ? warp - 2 : warp - C::W_DEC + 2) * 32 + lane;
      __half2 vsh[16];
      load_group_shift<Dv, NDT>(p.rsh + (size_t)hk * Dv, p.v_type, dt, vsh);
      int sk = 0, uk = 0, sv = 0, uv = 0;  // ring positions
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t & 1;
        const int j0 = (kt_begin + t) * BK + (int)rank * HK;  // first key of this CTA's half
        if (!wait_c(&bar[L_K_EMPTY + s], ((t >> 1) & 1) ^ 1)) break;
        const uint32_t kd = smem_u32(sK + s * C::KB), vd = smem_u32(sV + s * C::VB);
        for (int h = 0; h < EPT; ++h) {
          if (!(ok = wait(&bar[L_RK_FULL + sk], uk & 1))) break;
          const int nv = max(0, min(KE, p.M - (j0 + h * KE)));
          decode_rows<D, HK, NDT, false>(p.k_type, smem_u32(sRaw) + sk * kent, p.rbk_pad, KE, nv, h * KE, kd, st.sK,
                                         vsh, dt);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[L_RK_EMPTY + sk]);
          if (++sk == RK) sk = 0, ++uk;
        }
        if (!ok) break;
        fence_proxy_async_smem();  // the tile's binary16 stores, visible to the tensor cores
        __syncwarp();
        if (lane == 0) arrive_lead(L_K_FULL + s);
        if (!wait_c(&bar[L_V_EMPTY + s], ((t >> 1) & 1) ^ 1)) break;
        for (int h = 0; h < EPT; ++h) {
          if (!(ok = wait(&bar[L_RV_FULL + sv], uv & 1))) break;
          const int nv = max(0, min(KE, p.M - (j0 + h * KE)));
          decode_rows<Dv, HK, NDT, true>(p.v_type, smem_u32(sRawV) + sv * vent, p.rbv_pad, KE, nv, h * KE, vd, st.sV,
                                         vsh, dt);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[L_RV_EMPTY + sv]);
          if (++sv == RV) sv = 0, ++uv;
        }
        if (!ok) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) arrive_lead(L_V_FULL + s);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  {
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
      if (warp == 0 && lane == 0) {
        drain_loads(&bar[L_RK_FULL], RK, n_kraw, deadline);
        drain_loads(&bar[L_RV_FULL], RV, n_vraw, deadline);
      }
    }
    if (warp == 1 && lane == 0 && issued) mbar_wait_until(&bar[L_DRAIN], 0, deadline);
    // the issuer's last commits to this CTA's stage barriers (no one else waits for them).  After
    // an abort the tiles may not all have been issued; the products that were have landed once the
    // even CTA's issuer has seen L_DRAIN (its last commit, taken in order), before the cluster
    // barrier below that both CTAs pass before leaving
    if (warp == 2 && lane == 0 && !*s_abort) {
      for (int t = max(0, ntiles - 2); t < ntiles; ++t) {
        mbar_wait_until(&bar[L_K_EMPTY + (t & 1)], (t >> 1) & 1, deadline);
        mbar_wait_until(&bar[L_V_EMPTY + (t & 1)], (t >> 1) & 1, deadline);
      }
    }
  }
  // neither CTA frees its tensor memory or leaves while the other may still reach it
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, C::TCOLS);
  }
}

}  // namespace fab
