// Library-internal entry points shared by the translation units of libfa_back.so (hidden: not
// part of the C ABI in fa_back.h).
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "../../include/fa_back.h"

#ifdef __cplusplus
extern "C" {
#endif

// fa_back_workspace_size() for a plan restricted to at most ws_cap bytes of workspace where a
// cheaper key split would need more (the plan falls back to fewer key splits).
__attribute__((visibility("hidden"))) size_t fab_workspace_size_capped(int N, int M, int H, int Hkv, int D, int Dv,
                                                                       size_t ws_cap);

// Options of the backward beyond fa_back()'s arguments (NULL / 0 members: not used): the score
// extensions of fa_back_ext() and the plan restriction of fa_back_nocopy().
typedef struct fab_opts {
  const float* alibi;  // [H] ALiBi slopes
  float softcap;       // soft cap c (> 0), or 0
  const float* sinks;  // [H] sink logits
  float* dsinks;       // [H] sink-logit gradient (written when sinks is given), or NULL
  int nocopy;          // 1: only plans without the binary16 copy of the cache (levels 3 and 0)
} fab_opts;

// fa_back() with the same restriction on the plan.  With lse_in and delta_in (fa_back_with_stats)
// the row statistics are taken from them, the LSE pass is skipped and lse/delta may be null.
// With O (fa_forward) the call is the forward: dO, dQ, dK, dV, delta are null and lse, O written.
// ext (or NULL) adds the options of fa_back_ext() and fa_back_nocopy() to a plain backward.
__attribute__((visibility("hidden"))) fa_status fab_back_capped(
    const float* q, const void* k, int k_type, const void* v, int v_type, const uint16_t* mask, int mask_heads,
    const float* dO, float scale, int N, int M, int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK,
    float* dV, float* lse, float* delta, void* workspace, size_t workspace_bytes, void* stream, size_t ws_cap,
    const float* lse_in, const float* delta_in, float* O, const fab_opts* ext);

#ifdef __cplusplus
}
#endif
