// dQ as one product over the stored dS, with K decoded from the raw cache inside the CTA (the
// plan that stores dS but keeps no binary16 copy of the cache).
//
// A CTA owns two adjacent 128-row tiles of one KV head and one key split.  Per key tile it
// TMA-loads both row tiles' dS panels and the tile's raw K rows, decodes the rows once into a
// binary16 K' tile in shared memory, and issues dQ_a += dS_a K' for both row tiles a = 0, 1, with
// both 128 x D accumulators in tensor memory (2 D <= 512 columns).  Decoding each K tile once for
// 256 rows halves the decode work of a one-tile CTA, and the decode overlaps the stream of dS
// (read once, like k_dq_gemm's).
//
// Warp roles: 0 producer (dS panels and raw K rows; the whole warp for 4-byte copies), 1 tensor
// memory owner and MMA issuer, 2 .. 2+NDEC-1 decoders; warps 2-9 then read the accumulators out
// (warps 2-5 row tile 0, warps 6-9 row tile 1: every tensor-memory lane quarter twice).
#pragma once
#include "fa_kernels.cuh"

namespace fab {

template <int D, int BK>
struct DqRawCfg {
  static constexpr int NDEC = 12;  // a K tile's decode takes about as long as its two products
  static constexpr int NT = 32 * (2 + NDEC);
  static constexpr int AB = 128 * BK * 2;  // one row tile's dS panels for one key tile
  static constexpr int KB = BK * D * 2;    // binary16 K' tile
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_MAX = 232448;
  // dS stages: as many as leave room for two K' buffers and a raw ring of at least two 32-key
  // entries of the widest raw row of this head size (f32: 4 D bytes)
  static constexpr int RAW_MIN = 2 * 32 * 4 * D;
  static constexpr int NST_FIT = (SMEM_MAX - 1024 - 64 - BAR_BYTES - 2 * KB - RAW_MIN) / (2 * AB);
  static constexpr int NST = NST_FIT < 4 ? NST_FIT : 4;
  static constexpr int OFF_DS = 0;
  static constexpr int OFF_K = OFF_DS + NST * 2 * AB;
  static constexpr int OFF_BAR = OFF_K + 2 * KB;
  static constexpr int OFF_RAW = OFF_BAR + BAR_BYTES;
  static constexpr int RAW_BUDGET = SMEM_MAX - 1024 - 64 - OFF_RAW;
  static constexpr int TCOLS = pow2_at_least(2 * D);
  static_assert(NST >= 2, "shared memory budget");
  static_assert(TCOLS <= 512, "tensor memory budget");
  static_assert((NDEC * 32) % 64 == 0, "decoder_map needs a multiple of 8 column groups of 8 lanes");
};

enum {
  Q_RAW_FULL = 0,                             // [kMaxRawDepth] raw K entry landed
  Q_RAW_EMPTY = Q_RAW_FULL + kMaxRawDepth,    // [kMaxRawDepth] raw K entry decoded
  Q_DS_FULL = Q_RAW_EMPTY + kMaxRawDepth,     // [4] dS panels of both row tiles landed
  Q_DS_EMPTY = Q_DS_FULL + 4,                 // [4] their products done
  Q_K_FULL = Q_DS_EMPTY + 4,                  // [2] K' tile decoded
  Q_K_EMPTY = Q_K_FULL + 2,                   // [2] K' tile's products done
  Q_ACC_FULL = Q_K_EMPTY + 2,
  Q_COUNT
};
static_assert(8 * Q_COUNT + 8 <= 512, "barrier area");

template <int D, int BK>
static __global__ void __launch_bounds__(DqRawCfg<D, BK>::NT, 1)
    k_dq_raw(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmK, Params p) {
  using C = DqRawCfg<D, BK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sDS = sm + C::OFF_DS;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sRaw = sm + C::OFF_RAW;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * Q_COUNT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 8 * Q_COUNT + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt0 = 2 * blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int R = p.R, G = p.G;
  const int kt_begin = split * p.kt_per_split;
  const int kt_split_end = min(p.nKT, kt_begin + p.kt_per_split);
  // key tiles each row tile sees (the causal tail ends a row tile's keys at its last row's)
  int nt[2];
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int qt = qt0 + a;
    int kt_end = qt < p.nQT ? kt_split_end : kt_begin;
    if (p.causal && qt < p.nQT) {
      const long i_hi = (long)min(R - 1, qt * 128 + 127) / G;
      const long jmax = (long)p.M - p.N + i_hi;
      kt_end = min(kt_end, jmax < 0 ? 0 : (int)(jmax / BK) + 1);
    }
    nt[a] = max(0, kt_end - kt_begin);
  }
  const int ntiles = max(nt[0], nt[1]);
  const int KE = p.ke, EPT = BK / KE, RK = p.raw_depth;
  const int kent = KE * p.rbk_pad;  // bytes of one raw ring entry

  if (warp == 1) tmem_alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int s = 0; s < kMaxRawDepth; ++s) {
      mbar_init(&bar[Q_RAW_FULL + s], p.raw_bulk ? 1 : 32);
      mbar_init(&bar[Q_RAW_EMPTY + s], C::NDEC);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar[Q_DS_FULL + s], 1);
      mbar_init(&bar[Q_DS_EMPTY + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[Q_K_FULL + s], C::NDEC);
      mbar_init(&bar[Q_K_EMPTY + s], 1);
    }
    mbar_init(&bar[Q_ACC_FULL], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const Waiter wait{s_abort, p.err, p.wait_ns};
  int n_raw = 0, n_ds = 0;  // producer: raw entries and dS stages loaded

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmS);
      if (p.raw_bulk) prefetch_tmap(&tmK);
    }
    const int tot = ntiles * EPT;
    int e = 0, sr = 0, ur = 0, t = 0;
    uint64_t t0 = globaltimer_ns();
    while (e < tot || t < ntiles) {
      bool moved = false;
      int go_s = 0, go_r = 0;
      if (lane == 0) {
        go_s = t < ntiles && mbar_try_wait(&bar[Q_DS_EMPTY + t % C::NST], ((t / C::NST) & 1) ^ 1);
        go_r = e < tot && mbar_try_wait(&bar[Q_RAW_EMPTY + sr], (ur & 1) ^ 1);
      }
      go_s = __shfl_sync(0xffffffffu, go_s, 0);
      go_r = __shfl_sync(0xffffffffu, go_r, 0);
      if (go_s) {
        // both row tiles' dS panels of key tile t (a row tile past its keys loads nothing)
        if (lane == 0) {
          const int s = t % C::NST;
          uint64_t* fb = &bar[Q_DS_FULL + s];
          const uint32_t bytes = (uint32_t)(((t < nt[0]) ? C::AB : 0) + ((t < nt[1]) ? C::AB : 0));
          const int kt64 = (kt_begin + t) * (BK / 64);
          if (bytes) {
            mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              if (t >= nt[a]) continue;
#pragma unroll
              for (int c = 0; c < BK / 64; ++c)
                tma_load_3d(sDS + (s * 2 + a) * C::AB + c * (128 * 128), &tmS, fb, 0, 0,
                            (hk * p.nQT + qt0 + a) * p.ldds + kt64 + c);
            }
          } else {
            mbar_arrive(fb);
          }
        }
        __syncwarp();
        ++t, ++n_ds;
        moved = true;
      }
      if (go_r) {
        // raw K rows of entry e (keys ja .. ja+KE-1 of this head)
        const int ja = kt_begin * BK + e * KE;
        const int nv = max(0, min(KE, p.M - ja));
        uint64_t* fb = &bar[Q_RAW_FULL + sr];
        uint8_t* dst = sRaw + sr * kent;
        if (p.raw_bulk) {
          if (lane == 0) {
            if (nv > 0) {
              mbar_arrive_expect_tx(fb, (uint32_t)(KE * p.rbk));
              tma_load_3d(dst, &tmK, fb, 0, hk, ja);
            } else {
              mbar_arrive(fb);
            }
          }
        } else {
          const int w = p.rbk / 4;
          for (int x = lane; x < nv * w; x += 32) {
            const int rr = x / w, c = x % w;
            cp_async4(dst + rr * p.rbk_pad + 4 * c, p.k + ((size_t)(ja + rr) * p.Hkv + hk) * p.rbk + 4 * c);
          }
          cp_async_arrive(fb);
        }
        __syncwarp();
        ++e, ++n_raw;
        if (++sr == RK) sr = 0, ++ur;
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
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t ID = idesc_f16(128, D, false, true);
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % C::NST, kb = t & 1;
        if (!wait(&bar[Q_DS_FULL + s], (t / C::NST) & 1) || !wait(&bar[Q_K_FULL + kb], (t >> 1) & 1)) break;
        tc_fence_after();
        const uint64_t db = sdesc_sw128(smem_u32(sK + kb * C::KB), BK * 128, 1024);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          if (t >= nt[a]) continue;
          const uint64_t da = sdesc_sw128(smem_u32(sDS + (s * 2 + a) * C::AB), 16, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16(tbase + a * D, sdesc_adv(da, (k / 4) * (128 * 128) + (k % 4) * 32), sdesc_adv(db, k * 2048), ID,
                    (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&bar[Q_DS_EMPTY + s]);
        mma_commit(&bar[Q_K_EMPTY + kb]);
      }
      mma_commit(&bar[Q_ACC_FULL]);  // every product issued above (also after an abort)
    }
  } else {
    // ------------------------------------------------------------------ decoders, then epilogue
    constexpr int NDT = C::NDEC * 32;
    const int dt = (warp - 2) * 32 + lane;
    const float sigK = p.st->sK;  // K's operand scale
    __half2 nosh[16];  // K is not shifted: decode_rows<…, false> does not read these
    int sr = 0, ur = 0;
    bool ok = true;
    for (int t = 0; ok && t < ntiles; ++t) {
      const int kb = t & 1;
      const int j0 = (kt_begin + t) * BK;
      if (!wait(&bar[Q_K_EMPTY + kb], ((t >> 1) & 1) ^ 1)) break;
      const uint32_t kd = smem_u32(sK + kb * C::KB);
      for (int h = 0; h < EPT; ++h) {
        if (!(ok = wait(&bar[Q_RAW_FULL + sr], ur & 1))) break;
        const int nv = max(0, min(KE, p.M - (j0 + h * KE)));
        decode_rows<D, BK, NDT, false>(p.k_type, smem_u32(sRaw) + sr * kent, p.rbk_pad, KE, nv, h * KE, kd,
                                       sigK, nosh, dt);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[Q_RAW_EMPTY + sr]);
        if (++sr == RK) sr = 0, ++ur;
      }
      if (!ok) break;
      fence_proxy_async_smem();  // the tile's binary16 stores, visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[Q_K_FULL + kb]);
    }
    // epilogue: warps 2-5 read row tile 0's accumulator, warps 6-9 row tile 1's
    const int a = (warp - 2) >> 2;
    if (a < 2) {
      const int q4 = warp & 3;
      const int row = q4 * 32 + lane;
      const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
      const int qt = qt0 + a;
      const int r = qt * 128 + row;
      const bool rvalid = qt < p.nQT && r < R;
      const int i = rvalid ? r / G : 0;
      const int h = hk * G + (rvalid ? r % G : 0);
      float* out = !rvalid ? nullptr
                   : p.nsplit == 1 ? p.dQ + ((size_t)i * p.H + h) * D
                                   : p.dqpart + (((size_t)split * p.Hkv + hk) * R + r) * D;
      const Stats st = *p.st;
      const float dq_fac = !rvalid ? 0.f
                           : rows_need_own_scale(st) ? st.dq_fac * (st.lam / p.lamr[(size_t)hk * R + r])
                                                     : st.dq_fac;
      const bool have = (a ? nt[1] : nt[0]) > 0 && wait(&bar[Q_ACC_FULL], 0);
      if (have) tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float v[32];
        if (have) {
          tmem_ld32(tbase + a * D + lane_off + c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0.f;
        }
        if (out) {
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(out + c + x) =
                make_float4(v[x] * dq_fac, v[x + 1] * dq_fac, v[x + 2] * dq_fac, v[x + 3] * dq_fac);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*s_abort) {  // the same value in every thread: nothing writes it after the barrier
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    if (warp == 0 && lane == 0) {
      drain_loads(&bar[Q_RAW_FULL], RK, n_raw, deadline);
      drain_loads(&bar[Q_DS_FULL], C::NST, n_ds, deadline);
    }
    // the issuer committed every product it issued to Q_ACC_FULL before leaving its loop
    if (warp == 1 && lane == 0 && ntiles > 0) mbar_wait_until(&bar[Q_ACC_FULL], 0, deadline);
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

}  // namespace fab
