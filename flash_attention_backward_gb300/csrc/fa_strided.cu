// fa_back_strided(): the backward on inputs laid out as arbitrary views, and on a bit-packed mask.
//
// The operator keeps its outer strides and its q / dO component strides ("CUDA: FLASH_ATTN_BACK
// kernels", CambrianTech/llama.cpp pull request 63, PR description), and the raw-cache forward
// it sits beside reads a bit-packed mask ("chore(train): engine-10 continued", torad-labs/llama.cpp
// pull request 71, ncu tuning notes).  Here each strided input is gathered once into a contiguous
// region of the workspace and the mask's bits are widened to binary16 0 / -inf there; fa_back()
// then runs unchanged on those regions.  The gathers are HBM-bound copies: at the long-context
// shape Q, dO, K and V are 0.26 GB read and written once, about 0.08 ms at the copy rate against
// a 13.5 ms backward, and they keep every pass of the backward on its dense, TMA-friendly layout.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/fa_back.h"

namespace {

constexpr size_t kRegionAlign = 256;

size_t round_up(size_t x) { return (x + kRegionAlign - 1) / kRegionAlign * kRegionAlign; }

// Contiguous copies of the inputs at the front of the workspace; fa_back()'s own workspace follows.
struct Gathered {
  size_t off_q, off_do, off_k, off_v, off_mask, total;
};

Gathered layout(int N, int M, int H, int Hkv, int D, int Dv, long rbk, long rbv, int Hm) {
  Gathered g;
  size_t at = 0;
  g.off_q = at;
  at = round_up(at + (size_t)N * H * D * sizeof(float));
  g.off_do = at;
  at = round_up(at + (size_t)N * H * Dv * sizeof(float));
  g.off_k = at;
  at = round_up(at + (size_t)M * Hkv * rbk);
  g.off_v = at;
  at = round_up(at + (size_t)M * Hkv * rbv);
  g.off_mask = at;
  at = round_up(at + (size_t)Hm * N * M * sizeof(uint16_t));
  g.total = at;
  return g;
}

// dst row r holds source row (a, b), a = r / n1, b = r % n1: dst[r * n2 + c] = src[a * s0 + b * s1 +
// c * s2].  One warp per row, so one division per row; lanes walk c (coalesced where s2 = 1).
template <typename T>
__global__ void __launch_bounds__(256) k_gather_rows(T* __restrict__ dst, const T* __restrict__ src, long long n0,
                                                     long long n1, int n2, long long s0, long long s1, long long s2) {
  const long long rows = n0 * n1;
  const int lane = threadIdx.x & 31;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const long long a = r / n1, b = r - a * n1;
    const T* s = src + a * s0 + b * s1;
    T* d = dst + r * n2;
    for (int c = lane; c < n2; c += 32) d[c] = s[(long long)c * s2];
  }
}

// Bit-packed mask row (head a, query b) widened to binary16: key j is allowed (adds +0) when bit
// j % 32 of word j / 32 is set, masked (-inf, 0xFC00) when it is clear.
__global__ void __launch_bounds__(256) k_mask_bits(uint16_t* __restrict__ dst, const uint32_t* __restrict__ src,
                                                   long long n0, long long n1, int M, long long s0, long long s1) {
  const long long rows = n0 * n1;
  const int lane = threadIdx.x & 31;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const long long a = r / n1, b = r - a * n1;
    const uint32_t* s = src + a * s0 + b * s1;
    uint16_t* d = dst + r * M;
    for (int j = lane; j < M; j += 32) d[j] = ((s[j >> 5] >> (j & 31)) & 1u) ? (uint16_t)0x0000 : (uint16_t)0xFC00;
  }
}

unsigned gather_blocks(long long rows, int nsm) {
  // 8 rows (warps) a block; at most 8 blocks an SM, a whole number of waves over the SMs
  const long long want = (rows + 7) / 8;
  return (unsigned)std::max<long long>(1, std::min<long long>(want, 8LL * nsm));
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool head_size_supported(int d) { return d == 64 || d == 128 || d == 256; }

}  // namespace

extern "C" size_t fa_back_strided_workspace_size(int N, int M, int H, int Hkv, int D, int Dv, int k_type,
                                                 int v_type, int mask_heads) {
  const long rbk = fa_row_bytes(k_type, D), rbv = fa_row_bytes(v_type, Dv);
  if (rbk <= 0 || rbv <= 0 || N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv || mask_heads < 0) return 0;
  const size_t inner = fa_back_workspace_size(N, M, H, Hkv, D, Dv);
  if (inner == 0) return 0;
  return layout(N, M, H, Hkv, D, Dv, rbk, rbv, mask_heads).total + inner;
}

extern "C" fa_status fa_back_strided(const float* q, const void* k, int k_type, const void* v, int v_type,
                                     const void* mask, int mask_format, int mask_heads, const float* dO,
                                     const fa_strides* st, float scale, int N, int M, int H, int Hkv, int D, int Dv,
                                     int causal, float* dQ, float* dK, float* dV, float* lse, float* delta,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  // ---- argument checks (nothing is enqueued on failure); fa_back() repeats its own afterwards
  if (k_type < FA_F32 || k_type > FA_Q4_0 || v_type < FA_F32 || v_type > FA_Q4_0) return FA_ERR_TYPE;
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || Hkv > 256) return FA_ERR_SHAPE;
  if (mask && mask_heads != 1 && mask_heads != H) return FA_ERR_SHAPE;
  if (mask_format != FA_MASK_F16 && mask_format != FA_MASK_BITS) return FA_ERR_SHAPE;
  const long rbk = fa_row_bytes(k_type, D), rbv = fa_row_bytes(v_type, Dv);
  if (rbk <= 0 || rbv <= 0) return FA_ERR_SHAPE;
  if (!head_size_supported(D) || !head_size_supported(Dv)) return FA_ERR_UNSUPPORTED;
  if ((long)N * (H / Hkv) > (1L << 30) || M > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (!st) return FA_ERR_NULL;
  const long long strides[] = {st->q_row,  st->q_head, st->q_comp, st->do_row,    st->do_head, st->do_comp,
                               st->k_cell, st->k_head, st->v_cell, st->v_head,    st->mask_head, st->mask_row};
  for (long long s : strides)
    if (s < 0) return FA_ERR_SHAPE;
  const bool needQ = N > 0, needK = M > 0;
  if ((needQ && (!q || !dO || !dQ || !lse || !delta)) || (needK && (!k || !v || !dK || !dV))) return FA_ERR_NULL;
  // element alignment of the sources (the gathers move f32 words, 2-byte units of the cache
  // rows, and binary16 or 32-bit mask words); fa_back()'s 16-byte rule for the outputs
  if ((q && !aligned_to(q, 4)) || (dO && !aligned_to(dO, 4))) return FA_ERR_ALIGN;
  if ((k && !aligned_to(k, 2)) || (v && !aligned_to(v, 2))) return FA_ERR_ALIGN;
  if ((st->k_cell | st->k_head | st->v_cell | st->v_head) & 1) return FA_ERR_ALIGN;
  if (mask && !aligned_to(mask, mask_format == FA_MASK_BITS ? 4 : 2)) return FA_ERR_ALIGN;
  const void* outs[] = {dQ, dK, dV, lse, delta};
  for (const void* o : outs)
    if (o && !aligned_to(o, 16)) return FA_ERR_ALIGN;
  int dev = 0, nsm = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || nsm <= 0)
    return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;
  const int Hm = mask ? mask_heads : 0;
  const Gathered g = layout(N, M, H, Hkv, D, Dv, rbk, rbv, Hm);
  if (!workspace || workspace_bytes < g.total + fa_back_workspace_size_min(N, M, H, Hkv, D, Dv))
    return FA_ERR_WORKSPACE;
  if (!aligned_to(workspace, kRegionAlign)) return FA_ERR_ALIGN;

  // ---- gathers
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* q2 = reinterpret_cast<float*>(ws + g.off_q);
  float* do2 = reinterpret_cast<float*>(ws + g.off_do);
  uint8_t* k2 = ws + g.off_k;
  uint8_t* v2 = ws + g.off_v;
  uint16_t* m2 = reinterpret_cast<uint16_t*>(ws + g.off_mask);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (needQ) {
    const long long rows = (long long)N * H;
    k_gather_rows<float><<<gather_blocks(rows, nsm), 256, 0, s>>>(q2, q, N, H, D, st->q_row, st->q_head, st->q_comp);
    k_gather_rows<float><<<gather_blocks(rows, nsm), 256, 0, s>>>(do2, dO, N, H, Dv, st->do_row, st->do_head,
                                                                   st->do_comp);
  }
  if (needK) {
    const long long rows = (long long)M * Hkv;
    k_gather_rows<uint16_t><<<gather_blocks(rows, nsm), 256, 0, s>>>(
        reinterpret_cast<uint16_t*>(k2), static_cast<const uint16_t*>(k), M, Hkv, (int)(rbk / 2), st->k_cell / 2,
        st->k_head / 2, 1);
    k_gather_rows<uint16_t><<<gather_blocks(rows, nsm), 256, 0, s>>>(
        reinterpret_cast<uint16_t*>(v2), static_cast<const uint16_t*>(v), M, Hkv, (int)(rbv / 2), st->v_cell / 2,
        st->v_head / 2, 1);
  }
  if (mask && needQ && needK) {
    const long long rows = (long long)Hm * N;
    if (mask_format == FA_MASK_BITS)
      k_mask_bits<<<gather_blocks(rows, nsm), 256, 0, s>>>(m2, static_cast<const uint32_t*>(mask), Hm, N, M,
                                                             st->mask_head, st->mask_row);
    else
      k_gather_rows<uint16_t><<<gather_blocks(rows, nsm), 256, 0, s>>>(m2, static_cast<const uint16_t*>(mask), Hm,
                                                                       N, M, st->mask_head, st->mask_row, 1);
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

  // ---- the backward on the contiguous copies, with the rest of the workspace
  return fa_back(q2, k2, k_type, v2, v_type, mask ? m2 : nullptr, mask_heads, do2, scale, N, M, H, Hkv, D, Dv, causal,
                 dQ, dK, dV, lse, delta, ws + g.total, workspace_bytes - g.total, stream);
}
