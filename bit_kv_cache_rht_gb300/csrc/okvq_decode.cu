// Fused 2/4-bit decode attention ("OmniKVQuant: KV Cache Quantization for
// Omni-LLMs", section 1 INTRODUCTION, Implementation bullet: the quantized cache
// is unpacked inside attention without building a dense FP16 cache, the query is
// rotated once per head, and the inverse value rotations are batched after
// aggregation).
//
// decode_kernel - split-K over the token axis, one CTA per SM (12 warps at
//   2-bit, 8 at 4-bit). A CTA owns a range of 64-token pages of the flattened
//   (session, layer, kv head, page) list, cut into segments at unit boundaries
//   (the host balances pages plus a fixed cost per segment). A segment's
//   descriptor and queries are staged one segment ahead. Each warp streams whole
//   pages, one bulk copy each, into a private 2-stage shared-memory ring
//   (mbarrier completion, bounded waits) and works on 32-token half pages:
//     scores  S^T[16 x 8 tok] = [a_hi; a_lo][16 x 128] * Lambda^T[128 x 8 tok] + [beta; 0]
//             (mma m16n8k16; rows 0-7 / 8-15 = the 8 query heads' fp16 high and
//             residual parts of a = q' o range, so the sum is exact to ~2^-22)
//     softmax online, base 2, fp32 (m, l per head), lazy reference
//     values  O_m[128 ch x 8 heads] += Lcode[ch x 16 tok] * (p * n)[16 tok x 8 heads]
//   The score output fragment is already the value MMA's B fragment. Key and
//   value codes become fp16 MMA operands through a 64 KB shared-memory table
//   indexed by a whole code byte (built once per cache, bulk-copied per CTA);
//   one 8-byte load yields a whole operand register pair. One accumulator set
//   per modality in the rotated value domain: the current set in registers, the
//   others parked in tensor memory. Evicted tokens (page deletion masks) take no
//   part in the softmax. Warps merge through tensor memory (the warps of a lane
//   quarter) and shared memory (the four quarters); one partial (m, l, o_m) per
//   segment and head goes out; the merge kernel (okvq_combine.cu) combines them.
// lut_kernel - the code-byte -> fp16 level table, built once per cache.
#include "okvq_device.h"

namespace okvq {

namespace {

// warps 0-7 rotate query head w and build query fragment block w (8 blocks of 16 channels)
static_assert(MAXGQ == D / 16, "one warp per query head and per fragment block");
constexpr float INV_D = 1.0f / 128.0f;                      // (1/sqrt d) rotation * (1/sqrt d) softmax
constexpr int LUT_BYTES = 256 * 256;   // 256 code bytes x [K half | V half], 128 B each
constexpr float SOFTMAX_HEADROOM = 6.0f;   // log2 units
constexpr uint32_t TMEM_COLS = 512;        // parked modality accumulators: (warps / 4) x 3 x 32 columns

template <int BITS>
struct Cfg;
template <>
struct Cfg<2> {
  static constexpr int WARPS = 12;   // 3 per scheduler at 168 registers
  static constexpr int STAGES = 2;
  static constexpr bool QREG = true;  // query fragments held in registers for the whole segment
};
template <>
struct Cfg<4> {
  static constexpr int WARPS = 8;    // 9.4 KB pages: shared memory holds 8 warps x 2 stages
  static constexpr int STAGES = 2;
  static constexpr bool QREG = false;
};

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Tensor memory, 32 lanes x 32 columns of 32 bits per warp access (each lane its
// own row); warp-collective: every lane of the warp executes these.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[8][4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0][0]), "f"(v[0][1]), "f"(v[0][2]), "f"(v[0][3]), "f"(v[1][0]), "f"(v[1][1]), "f"(v[1][2]), "f"(v[1][3]),
      "f"(v[2][0]), "f"(v[2][1]), "f"(v[2][2]), "f"(v[2][3]), "f"(v[3][0]), "f"(v[3][1]), "f"(v[3][2]), "f"(v[3][3]),
      "f"(v[4][0]), "f"(v[4][1]), "f"(v[4][2]), "f"(v[4][3]), "f"(v[5][0]), "f"(v[5][1]), "f"(v[5][2]), "f"(v[5][3]),
      "f"(v[6][0]), "f"(v[6][1]), "f"(v[6][2]), "f"(v[6][3]), "f"(v[7][0]), "f"(v[7][1]), "f"(v[7][2]), "f"(v[7][3])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[8][4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0][0]), "=f"(v[0][1]), "=f"(v[0][2]), "=f"(v[0][3]), "=f"(v[1][0]), "=f"(v[1][1]), "=f"(v[1][2]),
        "=f"(v[1][3]), "=f"(v[2][0]), "=f"(v[2][1]), "=f"(v[2][2]), "=f"(v[2][3]), "=f"(v[3][0]), "=f"(v[3][1]),
        "=f"(v[3][2]), "=f"(v[3][3]), "=f"(v[4][0]), "=f"(v[4][1]), "=f"(v[4][2]), "=f"(v[4][3]), "=f"(v[5][0]),
        "=f"(v[5][1]), "=f"(v[5][2]), "=f"(v[5][3]), "=f"(v[6][0]), "=f"(v[6][1]), "=f"(v[6][2]), "=f"(v[6][3]),
        "=f"(v[7][0]), "=f"(v[7][1]), "=f"(v[7][2]), "=f"(v[7][3])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Per-warp value accumulators, one set per modality: the set of modality `cur`
// lives in registers, the others (once touched) wait in this warp's 32-column
// slots of tensor memory. Calls are warp-uniform.
struct ModAcc {
  uint32_t slot0;   // tensor-memory address of the modality-0 slot (this warp's lanes)
  int cur;          // modality held in registers, -1 none
  uint32_t live;    // modalities whose slot holds sums
};
__device__ __forceinline__ void mod_switch(ModAcc &ma, float (&acc)[8][4], int m) {
  if (ma.cur >= 0) {
    tmem_st32(ma.slot0 + 32u * (uint32_t)ma.cur, acc);
    ma.live |= 1u << ma.cur;
  }
  if ((ma.live >> m) & 1u) {
    tmem_ld32(ma.slot0 + 32u * (uint32_t)m, acc);
  } else {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  }
  ma.cur = m;
}
// scale the parked sets (head columns 2t4 / 2t4+1 by sf0 / sf1)
__device__ __forceinline__ void mod_rescale_parked(const ModAcc &ma, float sf0, float sf1) {
#pragma unroll 1
  for (int m = 0; m < MAXM; ++m) {
    if (m == ma.cur || !((ma.live >> m) & 1u)) continue;
    float v[8][4];
    tmem_ld32(ma.slot0 + 32u * (uint32_t)m, v);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      v[mt][0] *= sf0; v[mt][2] *= sf0;
      v[mt][1] *= sf1; v[mt][3] *= sf1;
    }
    tmem_st32(ma.slot0 + 32u * (uint32_t)m, v);
  }
}


__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// the level table lives at the start of dynamic shared memory; table reads are
// plain loads so the compiler can schedule them and fold the base address
__device__ __forceinline__ uint32_t lut32(const unsigned char *lut, uint32_t off) {
  return *reinterpret_cast<const uint32_t *>(lut + off);
}
__device__ __forceinline__ void lut64(const unsigned char *lut, uint32_t off, uint32_t &a, uint32_t &b) {
  const uint2 v = *reinterpret_cast<const uint2 *>(lut + off);
  a = v.x;
  b = v.y;
}

// shared-memory table address for code byte `B` (0..3) of word w:
// byte << 8 | lane part (laneoff holds it in its low byte)
template <int B>
__device__ __forceinline__ uint32_t lut_addr(uint32_t laneoff, uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(laneoff), "r"(w), "n"(0x1100u | ((4u + B) << 4)));
  return r;
}

// Cross-warp merge area of one segment (aliases the stage ring).
template <int WARPS>
struct Merge {
  float m[WARPS][MAXGQ];
  float l[WARPS][MAXGQ];
  float sc[WARPS][MAXGQ];        // exp2(m_w - M) per (warp, head)
  uint32_t held[WARPS];          // modalities each warp accumulated
  float q4[MAXM][4][32][32];     // per modality and lane quarter: the quarter's sum, [register][lane]
};

// value tile of one modality: acc[mt] += Lcode[16 ch x 16 tok] * P
template <int BITS>
__device__ __forceinline__ void value_mma(float (&acc)[8][4], const uint32_t *vw, const unsigned char *lut_v,
                                          uint32_t laneoff, uint32_t b0, uint32_t b1) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t A[4];
    if (BITS == 2) {
      const uint32_t w = vw[mt >> 1];
      const uint32_t a0 = (mt & 1) ? lut_addr<2>(laneoff, w) : lut_addr<0>(laneoff, w);
      const uint32_t a1 = (mt & 1) ? lut_addr<3>(laneoff, w) : lut_addr<1>(laneoff, w);
      lut64(lut_v, a0, A[0], A[1]);
      lut64(lut_v, a1, A[2], A[3]);
    } else {
      const uint32_t w = vw[mt];
      A[0] = lut32(lut_v, lut_addr<0>(laneoff, w));
      A[1] = lut32(lut_v, lut_addr<1>(laneoff, w));
      A[2] = lut32(lut_v, lut_addr<2>(laneoff, w));
      A[3] = lut32(lut_v, lut_addr<3>(laneoff, w));
    }
    mma16816(acc[mt], A, b0, b1);
  }
}

// key B fragments of one kb block for one 16-token tile:
// n-tile 0 (tokens 0-7): (pair 4kb, pair 4kb+2); n-tile 1: (pair 4kb+1, pair 4kb+3)
template <int BITS>
__device__ __forceinline__ void key_frags(const uint32_t *kw, int kb, const unsigned char *lut_k, uint32_t laneoff,
                                          uint32_t (&bf)[4]) {
  if (BITS == 2) {
    // one table entry = one B fragment: (pairs 4kb, 4kb+2), then (4kb+1, 4kb+3)
    const uint32_t w = kw[kb >> 1];
    const uint32_t a0 = (kb & 1) ? lut_addr<2>(laneoff, w) : lut_addr<0>(laneoff, w);
    const uint32_t a1 = (kb & 1) ? lut_addr<3>(laneoff, w) : lut_addr<1>(laneoff, w);
    lut64(lut_k, a0, bf[0], bf[1]);
    lut64(lut_k, a1, bf[2], bf[3]);
  } else {
    const uint32_t w = kw[kb];
    bf[0] = lut32(lut_k, lut_addr<0>(laneoff, w));
    bf[1] = lut32(lut_k, lut_addr<2>(laneoff, w));
    bf[2] = lut32(lut_k, lut_addr<1>(laneoff, w));
    bf[3] = lut32(lut_k, lut_addr<3>(laneoff, w));
  }
}

// Everything one warp needs to process 32-token half pages of one unit.
struct HalfPageCtx {
  const unsigned char *lut_k, *lut_v;
  const uint4 *qfrag;        // [8 kb][32 lanes]: (q_hi(ch 2t..), q_lo(ch 2t..), q_hi(ch 2t+8..), q_lo(..))
  const __half *qraw;        // [8][128] natural order
  const __half *tail;        // this unit's fp16 trailing keys
  const uint8_t *mod;        // this session's modality ids
  uint32_t laneoff;
  int T, Tf;
};

// One 32-token half page (two 16-token tiles) starting at page-relative token
// 32*hp of the staged page sp. FULLV: all 32 tokens exist and are quantized.
// SINGLE: every token of the page has modality ma.cur (checked by the caller).
// dead: the half page's deletion bits (bit i: token 32*hp + i was evicted); the
// caller guarantees at least one live token.
template <int BITS, int G, bool FULLV, bool SINGLE>
__device__ __forceinline__ void half_page(const HalfPageCtx &c, const PageLayout &PL, const unsigned char *sp,
                                          int tok0, int hp, uint32_t dead, float beta,
                                          float (&acc)[8][4], ModAcc &ma, float &m_run, float &l_run,
                                          const uint4 (&qreg)[8]) {
  constexpr int LANE_WORDS = BITS * 2;
  constexpr bool KT = G == 0;                 // TurboQuant keys: per-token norms, no groups
  constexpr int GG = KT ? PAGE : G;
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int hs = tok0 + 32 * hp;
  float sacc[4][4];                           // n-tiles (tile, nt); rows [hi | lo]
  if (FULLV || hs < c.Tf) {
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      sacc[n][0] = 0.f; sacc[n][1] = 0.f; sacc[n][2] = 0.f; sacc[n][3] = 0.f;
    }
    uint32_t kw[2][LANE_WORDS];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int i = 0; i < LANE_WORDS; i += 4) {
        const uint4 v4 =
            *reinterpret_cast<const uint4 *>(sp + (2 * hp + t) * PL.tile_bytes + lane * PL.lane_bytes + 4 * i);
        kw[t][i] = v4.x; kw[t][i + 1] = v4.y; kw[t][i + 2] = v4.z; kw[t][i + 3] = v4.w;
      }
    // a = q' o range of this half page's group as an exact fp16 pair (TwoProduct),
    // fragments [a_hi ; a_lo], built per 16-channel block right before its MMAs.
    // TurboQuant keys have no ranges: a = q' itself.
    const __half *rg = reinterpret_cast<const __half *>(sp + PL.off_stats + ((32 * hp) / GG) * 2 * D * 2 + D * 2);
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (!KT) v = *reinterpret_cast<const uint4 *>(rg + 32 * k2 + 8 * t4);
      const uint32_t rr[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int kb = 2 * k2 + u;
        const uint4 q = Cfg<BITS>::QREG ? qreg[kb] : c.qfrag[kb * 32 + lane];
        const uint32_t qh[2] = {q.x, q.z}, ql[2] = {q.y, q.w};
        uint32_t afk[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int h = 0; h < 2 && !KT; ++h) {
          const __half2 r2 = u2h(rr[2 * u + h]);
          const __half2 hi = __hmul2(u2h(qh[h]), r2);
          const __half2 er = __hfma2(u2h(qh[h]), r2, __hneg2(hi));
          const __half2 lo = __hfma2(u2h(ql[h]), r2, er);
          afk[2 * h] = h2u(hi);
          afk[2 * h + 1] = h2u(lo);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint32_t bf[4];
          key_frags<BITS>(kw[t], kb, c.lut_k, c.laneoff, bf);
          mma16816(sacc[2 * t + 0], afk, bf[0], bf[1]);
          mma16816(sacc[2 * t + 1], afk, bf[2], bf[3]);
        }
      }
    }
  } else {
    // trailing keys of an incomplete group: exact fp16 keys, unrotated query
    const int nt_valid = c.T - c.Tf;
#pragma unroll
    for (int n = 0; n < 4; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const int c0 = 16 * kb + 2 * t4;
      const uint32_t A[4] = {*reinterpret_cast<const uint32_t *>(c.qraw + g * D + c0), 0u,
                             *reinterpret_cast<const uint32_t *>(c.qraw + g * D + c0 + 8), 0u};
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int row = hs - c.Tf + 8 * n + g;
        const bool ok = row < nt_valid;
        const uint32_t b0 = ok ? *reinterpret_cast<const uint32_t *>(c.tail + row * D + c0) : 0u;
        const uint32_t b1 = ok ? *reinterpret_cast<const uint32_t *>(c.tail + row * D + c0 + 8) : 0u;
        mma16816(sacc[n], A, b0, b1);
      }
    }
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      sacc[n][0] *= LOG2E * INV_SQRT_D;
      sacc[n][1] *= LOG2E * INV_SQRT_D;
    }
  }
  // scores of head g for tokens hs + 8n + 2*t4 + e
  float s[4][2];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    // TurboQuant keys: k' = (n_t / sqrt d) l(code), so the token's norm scales its score
    float2 kn = make_float2(1.f, 1.f);
    if (KT)
      kn = __half22float2(*reinterpret_cast<const __half2 *>(sp + PL.off_stats + 2 * (32 * hp + 8 * n + 2 * t4)));
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      // the group offset joins after the MMA chain (it does not wait for it)
      const float v = KT ? (sacc[n][e] + sacc[n][2 + e]) * ((e ? kn.y : kn.x) * INV_SQRT_D)
                         : sacc[n][e] + sacc[n][2 + e] + ((FULLV || hs < c.Tf) ? beta : 0.f);
      s[n][e] = (FULLV || hs + 8 * n + 2 * t4 + e < c.T) ? v : -INFINITY;
    }
  }
  if (dead) {                                 // evicted tokens take no part in the softmax
    const uint32_t dl = dead >> (2 * t4);
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if ((dl >> (8 * n + e)) & 1u) s[n][e] = -INFINITY;
  }

  // ---- online softmax (base 2) for head g ----
  float mx = s[0][0];
#pragma unroll
  for (int n = 0; n < 4; ++n) mx = fmaxf(mx, fmaxf(s[n][0], s[n][1]));
  mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
  // lazy reference: m_run moves only when a score passes it, and then to the new
  // maximum plus headroom, so later small increases need no rescale; every
  // p = 2^(s - m_run) stays <= 1 and the largest stays >= 2^-headroom
  const bool up = mx > m_run;
  if (__any_sync(FULL, up)) {
    const float m_new = up ? mx + SOFTMAX_HEADROOM : m_run;
    const float sf = ex2(m_run - m_new);
    const float sf0 = __shfl_sync(FULL, sf, 8 * t4), sf1 = __shfl_sync(FULL, sf, 8 * t4 + 4);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc[mt][0] *= sf0; acc[mt][2] *= sf0;
      acc[mt][1] *= sf1; acc[mt][3] *= sf1;
    }
    if (ma.live & ~(ma.cur >= 0 ? 1u << ma.cur : 0u)) mod_rescale_parked(ma, sf0, sf1);
    l_run *= sf;
    m_run = m_new;
  }
  float p[4][2];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      p[n][e] = ex2(s[n][e] - m_run);
      l_run += p[n][e];
    }

  // ---- values, tile by tile ----
  const __half *norms = reinterpret_cast<const __half *>(sp + PL.off_norm);
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int tile = 2 * hp + t;
    const int ts = tok0 + 16 * tile;
    if (!FULLV && ts >= c.T) break;
    const int r0 = 16 * tile + 2 * t4;        // page-relative tokens r0, r0+1, r0+8, r0+9
    const float2 n01 = __half22float2(*reinterpret_cast<const __half2 *>(norms + r0));
    const float2 n89 = __half22float2(*reinterpret_cast<const __half2 *>(norms + r0 + 8));
    const bool v0 = FULLV || ts + 2 * t4 < c.T, v1 = FULLV || ts + 2 * t4 + 1 < c.T;
    const bool v8 = FULLV || ts + 2 * t4 + 8 < c.T, v9 = FULLV || ts + 2 * t4 + 9 < c.T;
    const float w0 = v0 ? p[2 * t][0] * n01.x : 0.f, w1 = v1 ? p[2 * t][1] * n01.y : 0.f;
    const float w8 = v8 ? p[2 * t + 1][0] * n89.x : 0.f, w9 = v9 ? p[2 * t + 1][1] * n89.y : 0.f;
    uint32_t vw[LANE_WORDS];
#pragma unroll
    for (int i = 0; i < LANE_WORDS; i += 4) {
      const uint4 v4 =
          *reinterpret_cast<const uint4 *>(sp + PL.off_v + tile * PL.tile_bytes + lane * PL.lane_bytes + 4 * i);
      vw[i] = v4.x; vw[i + 1] = v4.y; vw[i + 2] = v4.z; vw[i + 3] = v4.w;
    }
    if (SINGLE) {
      value_mma<BITS>(acc, vw, c.lut_v, c.laneoff, pack_h2(w0, w1), pack_h2(w8, w9));
      continue;
    }
    const uint32_t tmask = sp[PL.off_tmask + tile];
    if (__popc(tmask) == 1) {
      const int m = __ffs(tmask) - 1;
      if (m != ma.cur) mod_switch(ma, acc, m);
      value_mma<BITS>(acc, vw, c.lut_v, c.laneoff, pack_h2(w0, w1), pack_h2(w8, w9));
    } else {
      const uint8_t *modp = c.mod + ts + 2 * t4;
      const int m0 = v0 ? modp[0] : -1, m1 = v1 ? modp[1] : -1;
      const int m8 = v8 ? modp[8] : -1, m9 = v9 ? modp[9] : -1;
#pragma unroll
      for (int m = 0; m < MAXM; ++m) {
        if (!(tmask & (1u << m))) continue;
        const uint32_t b0 = pack_h2(m0 == m ? w0 : 0.f, m1 == m ? w1 : 0.f);
        const uint32_t b1 = pack_h2(m8 == m ? w8 : 0.f, m9 == m ? w9 : 0.f);
        if (m != ma.cur) mod_switch(ma, acc, m);
        value_mma<BITS>(acc, vw, c.lut_v, c.laneoff, b0, b1);
      }
    }
  }
}

// code byte -> fp16 level table; entry e = [K part 128 B | V part 128 B].
// 2-bit: byte = 2 pairs -> 8 B, replicated for the 16 lanes of a half warp;
// 4-bit: byte = 1 pair -> 4 B, replicated for 32 lanes. Built once per cache
// (lut_kernel) into global memory; each decode CTA bulk-copies it.
template <int BITS>
__global__ void lut_kernel(const LutArgs a) {
  unsigned char *lut = a.out;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 256 * 32; i += gridDim.x * blockDim.x) {
    const int e = i >> 5, c = i & 31;
    if (BITS == 2) {
      if (c >= 16) continue;
      const uint32_t k0 = h2u(__halves2half2(a.klev[e & 3], a.klev[(e >> 2) & 3]));
      const uint32_t k1 = h2u(__halves2half2(a.klev[(e >> 4) & 3], a.klev[(e >> 6) & 3]));
      const uint32_t v0 = h2u(__halves2half2(a.vlev[e & 3], a.vlev[(e >> 2) & 3]));
      const uint32_t v1 = h2u(__halves2half2(a.vlev[(e >> 4) & 3], a.vlev[(e >> 6) & 3]));
      *reinterpret_cast<uint2 *>(lut + e * 256 + c * 8) = make_uint2(k0, k1);
      *reinterpret_cast<uint2 *>(lut + e * 256 + 128 + c * 8) = make_uint2(v0, v1);
    } else {
      *reinterpret_cast<uint32_t *>(lut + e * 256 + c * 4) = h2u(__halves2half2(a.klev[e & 15], a.klev[e >> 4]));
      *reinterpret_cast<uint32_t *>(lut + e * 256 + 128 + c * 4) =
          h2u(__halves2half2(a.vlev[e & 15], a.vlev[e >> 4]));
    }
  }
}

// The rare partial half pages (a unit's last page, pages with evicted tokens) run
// out of line, so the common path's code stays small.
struct TailState {
  float acc[8][4];
  ModAcc ma;
  float m_run, l_run;
  uint4 qreg[8];
  HalfPageCtx hc;
};
template <int BITS, int G, bool SINGLE>
__device__ __noinline__ void half_page_partial(TailState *ts, const unsigned char *sp, int tok0, int hp, uint32_t dead,
                                               float beta) {
  const PageLayout PL = page_layout(BITS, G);
  half_page<BITS, G, false, SINGLE>(ts->hc, PL, sp, tok0, hp, dead, beta, ts->acc, ts->ma, ts->m_run, ts->l_run,
                                    ts->qreg);
}
template <int BITS, int G, bool SINGLE>
__device__ __forceinline__ void call_partial(const HalfPageCtx &hc, const unsigned char *sp, int tok0, int hp,
                                             uint32_t dead, float beta, float (&acc)[8][4], ModAcc &ma,
                                             float &m_run, float &l_run, const uint4 (&qreg)[8]) {
  TailState ts;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) ts.acc[i][j] = acc[i][j];
    ts.qreg[i] = qreg[i];
  }
  ts.ma = ma;
  ts.m_run = m_run;
  ts.l_run = l_run;
  ts.hc = hc;
  half_page_partial<BITS, G, SINGLE>(&ts, sp, tok0, hp, dead, beta);
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = ts.acc[i][j];
  ma = ts.ma;
  m_run = ts.m_run;
  l_run = ts.l_run;
}

// The cross-warp merge of one segment, after every warp parked its modality sums
// in tensor memory and wrote its (m, l) and held set: per-(warp, head) scales
// (threads 0-7, which also write the partial's m and l), then the sums of each
// lane quarter's warps (w, w + 4, w + 8 share tensor-memory rows) in tensor
// memory, then the four quarter sums in shared memory, lane-major. Out of line:
// its registers stay out of the page loop's allocation.
template <int WARPS>
__device__ __noinline__ void segment_merge(Merge<WARPS> *MG, float *part, uint32_t tbase, int nmod) {
  constexpr int THREADS = WARPS * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, t4 = lane & 3;
  // per-(warp, head) scales, once
  if (tid < MAXGQ) {
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, MG->m[w][tid]);
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float sc = MG->m[w][tid] == -INFINITY ? 0.f : ex2(MG->m[w][tid] - M);
      MG->sc[w][tid] = sc;
      L += sc * MG->l[w][tid];
    }
    part[tid * PARTIAL_FLOATS + 0] = M;
    part[tid * PARTIAL_FLOATS + 1] = L;
  }
  __syncthreads();
  // warps of one lane quarter (w, w + 4, w + 8) share their tensor-memory rows:
  // warp w sums, for modality m = w / 4 (+ WARPS / 4 ...), the scaled sets of its
  // quarter; the four quarter sums meet in shared memory, lane-major
  float *R4 = &MG->q4[0][0][0][0];
  {
    const int q = warp & 3;
#pragma unroll 1
    for (int m = warp >> 2; m < nmod; m += WARPS / 4) {
      float sum[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) sum[mt][0] = sum[mt][1] = sum[mt][2] = sum[mt][3] = 0.f;
#pragma unroll 1
      for (int k = 0; k < WARPS / 4; ++k) {
        const int src = q + 4 * k;
        if (!((MG->held[src] >> m) & 1u)) continue;   // warp-uniform
        float v[8][4];
        tmem_ld32(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(k * MAXM * 32 + 32 * m), v);
        const float s0 = MG->sc[src][2 * t4], s1 = MG->sc[src][2 * t4 + 1];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          sum[mt][0] = fmaf(s0, v[mt][0], sum[mt][0]);
          sum[mt][1] = fmaf(s1, v[mt][1], sum[mt][1]);
          sum[mt][2] = fmaf(s0, v[mt][2], sum[mt][2]);
          sum[mt][3] = fmaf(s1, v[mt][3], sum[mt][3]);
        }
      }
      float *dst = R4 + (size_t)(m * 4 + q) * 32 * 32 + lane;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[(4 * mt + e) * 32] = sum[mt][e];
    }
  }
  tc_fence_before();                             // the slot reads are done before the next segment parks
  __syncthreads();
  tc_fence_after();
  // register i = 4 mt + e of lane (g, t4): head 2 t4 + (e & 1), channel 16 mt + g + 8 (e >> 1)
  for (int idx = tid; idx < nmod * 32 * 32; idx += THREADS) {
    const int m = idx >> 10, i = (idx >> 5) & 31, ln = idx & 31;
    const float *r = R4 + (size_t)m * 4 * 32 * 32 + i * 32 + ln;
    const float o = (r[0] + r[32 * 32]) + (r[2 * 32 * 32] + r[3 * 32 * 32]);
    const int head = 2 * (ln & 3) + (i & 1), ch = 16 * (i >> 2) + (ln >> 2) + 8 * ((i >> 1) & 1);
    part[head * PARTIAL_FLOATS + 2 + m * D + ch] = o;
  }
}

template <int BITS, int G>
__global__ void __launch_bounds__(Cfg<BITS>::WARPS * 32, 1) decode_kernel(const DecodeArgs a) {
  constexpr int WARPS = Cfg<BITS>::WARPS;
  constexpr int THREADS = WARPS * 32;
  static_assert(WARPS >= MAXGQ && WARPS % 4 == 0 && (WARPS / 4) * MAXM * 32 <= TMEM_COLS, "warp layout");
  constexpr int STAGES = Cfg<BITS>::STAGES;
  constexpr int LANE_WORDS = BITS * 2;        // 32-bit words per lane chunk
  const PageLayout PL = page_layout(BITS, G);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *lut = smem;                                            // LUT_BYTES
  float *qr = reinterpret_cast<float *>(smem + LUT_BYTES);              // [8][128] stat order, scaled
  __half *qraw = reinterpret_cast<__half *>(qr + MAXGQ * D);            // [8][128] natural order
  __half *qstage = qraw + MAXGQ * D;                                    // [8][128] next segment's queries
  uint4 *qfrag = reinterpret_cast<uint4 *>(qstage + MAXGQ * D);         // [8 kb][32 lanes]
  uint64_t *bars = reinterpret_cast<uint64_t *>(qfrag + 8 * 32);        // [WARPS][STAGES]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + WARPS * STAGES);
  // 128-byte aligned stage ring, as an offset from the (aligned) shared base: a round
  // trip through an integer would hide that these are shared-memory addresses
  const size_t stage_off = (reinterpret_cast<unsigned char *>(tmem_slot + 4) - smem + 127) & ~size_t(127);
  unsigned char *stages = smem + stage_off;
  Merge<WARPS> &MG = *reinterpret_cast<Merge<WARPS> *>(stages);
  unsigned char *my_stage0 = stages + (size_t)warp * STAGES * PL.page_bytes;
  uint64_t *my_bars = bars + warp * STAGES;

  // the level table (built once per cache) arrives by one bulk copy; it is first
  // needed after the first segment's query rotation
  __shared__ __align__(8) uint64_t lut_bar;
  // the next segment's descriptor and queries (bulk copy) are staged while the
  // current one runs, so a segment starts without global latency
  __shared__ __align__(8) uint64_t q_bar;
  __shared__ int sd_unit, sd_pb, sd_pe, sd_tail, sd_slot;
  __shared__ int cur_slot;    // the running segment's partial slot, read by its merge
  // the Hadamard signs (written at create), staged before the dependency wait
  __shared__ __align__(16) float sgn[D];
  __shared__ long long sd_T;
  const int gq = a.Hq / a.Hkv;
  struct SegDesc {
    int unit, pb, pe, slot, tail;
    long long T;
  };
  auto load_desc = [&](int sg) {
    SegDesc d;
    d.unit = a.segs[4 * sg + 0];
    d.pb = a.segs[4 * sg + 1];
    d.pe = a.segs[4 * sg + 2];
    d.slot = a.segs[4 * sg + 3];
    d.T = a.unit_len[d.unit];
    d.tail = a.unit_tail[d.unit];
    return d;
  };
  auto stage_segment = [&](const SegDesc &d) {  // one thread
    sd_unit = d.unit;
    sd_pb = d.pb;
    sd_pe = d.pe;
    sd_slot = d.slot;
    sd_T = d.T;
    sd_tail = d.tail;
    const int ss = d.unit / (a.L * a.Hkv), lh = d.unit % (a.L * a.Hkv);
    const __half *qsrc = a.q + (((long long)ss * a.L + lh / a.Hkv) * a.Hq + (long long)(lh % a.Hkv) * gq) * D;
    fence_async_smem();
    bulk_load(qstage, qsrc, (uint32_t)(gq * D * sizeof(__half)), &q_bar);
  };
  // Launched as a programmatic dependent of the previous kernel on the stream (the
  // last step's merge): everything up to griddepcontrol.wait reads only the cache's
  // level table and Hadamard signs (written at create) and the work list (written by
  // a host copy that the launch itself follows); queries and pages come after it.
  const int seg_begin = a.cta_seg[blockIdx.x], seg_end = a.cta_seg[blockIdx.x + 1];
  SegDesc first{};
  if (tid == 0 && seg_begin < seg_end) first = load_desc(seg_begin);
  if (tid == 0) {
    mbar_init(&lut_bar, 1);
    mbar_init(&q_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    bulk_load(lut, a.lut, LUT_BYTES, &lut_bar);
  }
  if (lane == 0)
    for (int s = 0; s < STAGES; ++s) mbar_init(&my_bars[s], 1);
  if (tid < D / 4) reinterpret_cast<float4 *>(sgn)[tid] = reinterpret_cast<const float4 *>(a.signs)[tid];
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // tensor memory for the parked modality accumulators: 2 warps per lane quarter,
  // 3 x 32 columns each
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the merge kernel may be scheduled as SMs free up; it waits for this grid's memory
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0 && seg_begin < seg_end) stage_segment(first);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t slot0 = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(warp >> 2) * (MAXM * 32);

  const unsigned char *lut_k = lut, *lut_v = lut + 128;
  const uint32_t laneoff = BITS == 2 ? (uint32_t)((lane & 15) << 3) : (uint32_t)(lane << 2);
  int ring_st = 0;          // stage of the next page this warp consumes
  uint32_t ring_par = 0;    // its mbarrier phase parity
  bool wait_failed = false;
  bool lut_ready = false;

  int seg = seg_begin;
  for (; seg < seg_end; ++seg) {
    const int unit = sd_unit;
    const int pb = sd_pb, pe = sd_pe;
    const int session = unit / (a.L * a.Hkv);
    const int T = (int)sd_T;
    const int tail_sel = sd_tail;
    if (tid == 0) cur_slot = sd_slot;     // before the stager overwrites sd_* (barriers below)
    // the next segment's descriptor: loaded now by a thread whose warp has no head
    // to rotate (at 2-bit), staged with its queries once the rotation is done
    const bool stager = tid == THREADS - 32 && seg + 1 < seg_end;
    SegDesc next{};
    if (stager) next = load_desc(seg + 1);
    constexpr bool KT = G == 0;               // TurboQuant keys: all quantized, no groups
    constexpr int GG = KT ? PAGE : G;
    const int Tf = KT ? T : (T / GG) * GG;
    const unsigned char *unit_pages = a.pages + (long long)unit * a.P_max * PL.page_bytes;
    const __half *tail = a.tails + ((long long)tail_sel * a.units + unit) * (long long)G * D;
    // each warp's first page is on its way while the query is rotated (the ring is
    // free: the previous segment's merge ended with a barrier)
    const int npages = pe - pb;
    const int my_n = npages > warp ? (npages - warp + WARPS - 1) / WARPS : 0;
    if (lane == 0) {
      for (int k = 0; k < min(my_n, 1); ++k) {
        const int st = (ring_st + k) % STAGES;
        fence_async_smem();
        bulk_load(my_stage0 + (size_t)st * PL.page_bytes,
                  unit_pages + (long long)(pb + warp + k * WARPS) * PL.page_bytes, PL.page_bytes, &my_bars[st]);
      }
    }

    // ---- rotate the query group once: q' = H (s o q) / d, in log2 units (warp = head) ----
    if (!mbar_wait(&q_bar, (uint32_t)(seg - seg_begin) & 1u)) wait_failed = true;
    if (warp < MAXGQ) {
      const int hh = warp;
      float x[4];
      const float4 sg4 = reinterpret_cast<const float4 *>(sgn)[lane];
      const float sg[4] = {sg4.x, sg4.y, sg4.z, sg4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 4 * lane + j;
        const __half hv = hh < gq ? qstage[hh * D + c] : __float2half(0.f);
        qraw[hh * D + c] = hv;
        x[j] = __half2float(hv) * sg[j];
      }
      float y0 = x[0] + x[1], y1 = x[0] - x[1], y2 = x[2] + x[3], y3 = x[2] - x[3];
      x[0] = y0 + y2; x[2] = y0 - y2; x[1] = y1 + y3; x[3] = y1 - y3;
#pragma unroll
      for (int sm = 1; sm < 32; sm <<= 1) {
        const bool upper = (lane & sm) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = __shfl_xor_sync(FULL, x[j], sm);
          x[j] = upper ? p - x[j] : x[j] + p;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 4 * lane + j;
        qr[hh * D + stat_pos(c)] = x[j] * (INV_D * LOG2E);
      }
    }
    __syncthreads();

    // query fragments for the score and offset MMAs, one kb block per warp:
    // lane (g, t4) gets head g, channels 16kb + 2t4 + {0,1} and + 8 + {0,1}, fp16 high + residual
    if (warp < D / 16) {
      const int kb = warp;
      const float4 v = *reinterpret_cast<const float4 *>(qr + g * D + 32 * (kb >> 1) + 8 * t4 + 4 * (kb & 1));
      const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      qfrag[kb * 32 + lane] = make_uint4(h2u(h01), pack_h2(v.x - f01.x, v.y - f01.y), h2u(h23),
                                         pack_h2(v.z - f23.x, v.w - f23.y));
    }
    __syncthreads();
    // the descriptor and queries of this CTA's next segment, staged while this one runs
    if (stager) stage_segment(next);
    // the rest of the ring: one page per warp went out first, so that the first
    // pages of all warps arrive before any second page competes with them
    if (lane == 0) {
      for (int k = 1; k < min(my_n, STAGES); ++k) {
        const int st = (ring_st + k) % STAGES;
        fence_async_smem();
        bulk_load(my_stage0 + (size_t)st * PL.page_bytes,
                  unit_pages + (long long)(pb + warp + k * WARPS) * PL.page_bytes, PL.page_bytes, &my_bars[st]);
      }
    }

    HalfPageCtx hc;
    hc.lut_k = lut_k;
    hc.lut_v = lut_v;
    hc.qfrag = qfrag;
    uint4 qreg[8];             // this lane's query fragments (registers when Cfg::QREG)
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) qreg[kb] = Cfg<BITS>::QREG ? qfrag[kb * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
    hc.qraw = qraw;
    hc.tail = tail;
    hc.mod = a.mod + (long long)session * a.cap;
    hc.laneoff = laneoff;
    hc.T = T;
    hc.Tf = Tf;

    // ---- per-warp state ----
    float acc[8][4];         // value sums of modality ma.cur (the others parked in tensor memory)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    ModAcc ma{slot0, -1, 0u};
    float m_run = -INFINITY, l_run = 0.f;     // head g

    if (!lut_ready) {                         // once: the bulk copy of the level table
      if (!mbar_wait(&lut_bar, 0u)) wait_failed = true;
      lut_ready = true;
    }

    for (int k = 0; k < my_n; ++k) {
      const int st = ring_st;
      if (!mbar_wait(&my_bars[st], ring_par)) {
        wait_failed = true;
        break;
      }
      if (++ring_st == STAGES) {
        ring_st = 0;
        ring_par ^= 1u;
      }
      __syncwarp();
      const unsigned char *sp = my_stage0 + (size_t)st * PL.page_bytes;
      const int page = pb + warp + k * WARPS;
      const int tok0 = page * PAGE;

      // group offsets beta(head g, group) = q' . min for the page's groups (tensor cores)
      float beta_g0 = 0.f, beta_g1 = 0.f;
      if (!KT && tok0 < Tf) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          uint32_t b0 = 0u, b1 = 0u;
          if (g < PAGE / GG) {
            const __half *mn = reinterpret_cast<const __half *>(sp + PL.off_stats + g * 2 * D * 2);
            const uint2 v = *reinterpret_cast<const uint2 *>(mn + 32 * (kb >> 1) + 8 * t4 + 4 * (kb & 1));
            b0 = v.x;
            b1 = v.y;
          }
          const uint4 q = Cfg<BITS>::QREG ? qreg[kb] : qfrag[kb * 32 + lane];
          const uint32_t A[4] = {q.x, q.y, q.z, q.w};
          mma16816(d, A, b0, b1);
        }
        beta_g0 = __shfl_sync(FULL, d[0] + d[2], 4 * g);
        beta_g1 = __shfl_sync(FULL, d[1] + d[3], 4 * g);
      }

      // modalities present in the page: one (the common case) runs without per-tile checks
      const uint32_t tmw = *reinterpret_cast<const uint32_t *>(sp + PL.off_tmask);
      const unsigned long long dead = *reinterpret_cast<const unsigned long long *>(sp + PL.off_tmask + DEAD_OFF);
      const uint32_t pmask = (tmw | (tmw >> 8) | (tmw >> 16) | (tmw >> 24)) & 0xFFu;
      const bool single = __popc(pmask) == 1;
      if (single && __ffs(pmask) - 1 != ma.cur) mod_switch(ma, acc, __ffs(pmask) - 1);
#pragma unroll 1
      for (int hp = 0; hp < 2; ++hp) {
        const int hs = tok0 + 32 * hp;
        if (hs >= T) break;
        const uint32_t dh = (uint32_t)(dead >> (32 * hp));
        if (dh) {                                 // evicted tokens: skip the half page if none is live
          const int nv = min(32, T - hs);
          if (!((nv >= 32 ? 0xFFFFFFFFu : (1u << nv) - 1u) & ~dh)) continue;
        }
        const float beta = (G == 32 && hp == 1) ? beta_g1 : beta_g0;
        const bool full = hs + 32 <= Tf;
        if (single) {
          if (full)
            half_page<BITS, G, true, true>(hc, PL, sp, tok0, hp, dh, beta, acc, ma, m_run, l_run, qreg);
          else
            call_partial<BITS, G, true>(hc, sp, tok0, hp, dh, beta, acc, ma, m_run, l_run, qreg);
        } else {
          if (full)
            half_page<BITS, G, true, false>(hc, PL, sp, tok0, hp, dh, beta, acc, ma, m_run, l_run, qreg);
          else
            call_partial<BITS, G, false>(hc, sp, tok0, hp, dh, beta, acc, ma, m_run, l_run, qreg);
        }
      }
      __syncwarp();
      // refill this stage with the page STAGES ahead
      if (lane == 0 && k + STAGES < my_n) {
        fence_async_smem();
        bulk_load(my_stage0 + (size_t)st * PL.page_bytes,
                  unit_pages + (long long)(pb + warp + (k + STAGES) * WARPS) * PL.page_bytes, PL.page_bytes,
                  &my_bars[st]);
      }
    }
    if (__syncthreads_or(wait_failed)) {
      // a copy never completed: report it, give copies still in flight a bounded
      // chance to land, and leave this CTA's partials unwritten
      if (tid == 0) atomicOr(a.err, ERR_WAIT);
      if (lane == 0)
        for (int s2 = 0; s2 < STAGES; ++s2) (void)mbar_wait(&my_bars[(ring_st + s2) % STAGES], ring_par ^ (s2 + ring_st >= STAGES ? 1u : 0u));
      break;
    }

    // ---- per-warp totals: head g lives in lanes 4g..4g+3 ----
    l_run += __shfl_xor_sync(FULL, l_run, 1);
    l_run += __shfl_xor_sync(FULL, l_run, 2);
    const uint32_t held = ma.live | (ma.cur >= 0 ? 1u << ma.cur : 0u);
    if (t4 == 0) {
      MG.m[warp][g] = m_run;
      MG.l[warp][g] = l_run;
    }
    if (lane == 0) MG.held[warp] = held;
    // every modality sum of this warp goes to (or stays in) its tensor-memory slots
    if (ma.cur >= 0) tmem_st32(ma.slot0 + 32u * (uint32_t)ma.cur, acc);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    segment_merge<WARPS>(&MG, a.partials + (long long)cur_slot * MAXGQ * PARTIAL_FLOATS, tbase, a.M);
    __syncthreads();              // merge area is the stage ring of the next segment
  }
  // the level table's and a staged query copy must land before the CTA's shared
  // memory goes away (one is left unconsumed when the loop ended early)
  if (!lut_ready && tid == 0 && !mbar_wait(&lut_bar, 0u)) atomicOr(a.err, ERR_WAIT);
  if (seg < seg_end && tid == 0)
    for (int s2 = seg; s2 < min(seg + 2, seg_end); ++s2)
      if (!mbar_wait(&q_bar, (uint32_t)(s2 - seg_begin) & 1u)) atomicOr(a.err, ERR_WAIT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(TMEM_COLS));
  }
}

template <int BITS, int G>
cudaError_t launch_decode_t(const DecodeArgs &a, int n_cta, cudaStream_t s) {
  static std::atomic<uint64_t> attr_done{0};
  const size_t smem = decode_smem_bytes(BITS, G);
  cudaError_t e = once_per_device(attr_done, [&] {
    return cudaFuncSetAttribute(decode_kernel<BITS, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_cta);
  cfg.blockDim = dim3(Cfg<BITS>::WARPS * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<BITS, G>, a);
}

}  // namespace

template <int BITS>
size_t decode_smem_bytes_t(int G) {
  const PageLayout PL = page_layout(BITS, G);
  constexpr int W = Cfg<BITS>::WARPS, STAGES = Cfg<BITS>::STAGES;
  size_t head = LUT_BYTES + MAXGQ * D * 4 + 2 * MAXGQ * D * 2 + 8 * 32 * 16 + W * STAGES * 8 + 16;
  size_t ring = (size_t)W * STAGES * PL.page_bytes;
  if (ring < sizeof(Merge<W>)) ring = sizeof(Merge<W>);
  return head + 128 + ring;
}

cudaError_t launch_lut(int bits, const LutArgs &a, cudaStream_t s) {
  if (bits == 2) lut_kernel<2><<<32, 256, 0, s>>>(a);
  else lut_kernel<4><<<32, 256, 0, s>>>(a);
  return cudaGetLastError();
}

int decode_warps(int bits) { return bits == 2 ? Cfg<2>::WARPS : Cfg<4>::WARPS; }

size_t decode_smem_bytes(int bits, int G) { return bits == 2 ? decode_smem_bytes_t<2>(G) : decode_smem_bytes_t<4>(G); }

cudaError_t launch_decode(const DecodeArgs &a, int n_cta, cudaStream_t s) {
  if (n_cta <= 0) return cudaSuccess;
  if (a.G == 0) return a.bits == 2 ? launch_decode_t<2, 0>(a, n_cta, s) : launch_decode_t<4, 0>(a, n_cta, s);
  if (a.bits == 2 && a.G == 32) return launch_decode_t<2, 32>(a, n_cta, s);
  if (a.bits == 2 && a.G == 64) return launch_decode_t<2, 64>(a, n_cta, s);
  if (a.bits == 4 && a.G == 32) return launch_decode_t<4, 32>(a, n_cta, s);
  return launch_decode_t<4, 64>(a, n_cta, s);
}

}  // namespace okvq
