// Append launch interface of libokvq (the host API and the append kernels): the
// arguments of one okvq_append_chunk and the launcher of its two grids.
#pragma once
#include "okvq_internal.h"

namespace okvq {

constexpr int V_MAX_PPC = 32;      // pages one CTA of the value append takes at most
constexpr int MAX_G = 64;          // largest key group (group sizes are 32 or 64)

struct AppendArgs {
  const __half *k;          // [n][L][Hkv][D]
  const __half *v;
  const uint8_t *mod_in;    // [n]
  int n;                    // tokens in this chunk
  long long T0;             // session length before the append
  int session;
  int L, Hkv, M, bits, G;   // G: key group size, 0 = TurboQuant keys (per-token norms)
  long long P_max;
  uint8_t *pages;           // all units
  __half *tail_old;         // [units][G][D] buffer read (current)
  __half *tail_new;         // [units][G][D] buffer written (next)
  uint8_t *mod;             // [S][cap] session modality ids
  long long cap;            // max_tokens rounded up to a page
  const __half *rot_h;      // [L][Hkv][M][2][D][D]: R[i][c] as fp16 high, then residual part
  const float *signs;       // [D] +-1 Hadamard signs
  uint32_t *err;
  long long page0;          // first page touched
  int vppc;                 // pages per CTA of the value kernel (1 .. V_MAX_PPC)
  int vwide;                // 1: two value CTAs per SM (their register budget), 0: one
  int nlev;
  float vthr[15];           // fp32 value thresholds (midpoints of the fp16 levels)
  float kthr[15];           // fp32 key thresholds (midpoints of the fp16 key levels)
};

cudaError_t launch_append(const AppendArgs &a, int n_pages, cudaStream_t s, cudaStream_t aux, cudaEvent_t fork,
                          cudaEvent_t join);

}  // namespace okvq
