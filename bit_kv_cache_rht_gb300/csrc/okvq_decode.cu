// Fused 2/4-bit decode attention ("OmniKVQuant: KV Cache Quantization for
// Omni-LLMs", section 1 INTRODUCTION, Implementation bullet: the quantized cache
// is unpacked inside attention without building a dense FP16 cache, the query is
// rotated once per head, and the inverse value rotations are batched after
// aggregation).
//
// decode_kernel - split-K over the token axis. A CTA (4 warps) owns a balanced
//   range of 64-token pages of the flattened (session, layer, kv head, page)
//   list, cut into segments at unit boundaries. Each warp streams whole pages
//   with one bulk copy each into a private shared-memory ring (mbarrier
//   completion), and for every 16-token tile runs
//     scores  S[16 tok x 8 heads] = beta_g + Lambda[tok x 128] * (q' o (mx-mn))   (mma m16n8k16)
//     softmax online, base 2, fp32 (m, l per head)
//     values  O_m[128 ch x 8 heads] += Lcode[ch x tok] * (p * n)[tok x heads]     (mma m16n8k16)
//   with the code -> fp16 level lookups done in registers from shared tables,
//   one accumulator set per modality (rotated value domain). Warps merge in
//   shared memory; one partial (m, l, o_m) per segment and head goes to global.
// combine_kernel - per (unit, 32 output channels): log-sum-exp merge of the
//   unit's partials, O = (sum_m R_m^T o_m) / (l sqrt d), fp16 store.
#include "okvq_internal.h"

namespace okvq {

namespace {

constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr float LOG2E = 1.4426950408889634074f;
constexpr float INV_D = 1.0f / 128.0f;                      // (1/sqrt d) rotation * (1/sqrt d) softmax
constexpr float INV_SQRT_D = 0.0883883476483184405501f;
constexpr unsigned FULL = 0xffffffffu;
constexpr long long WAIT_LIMIT = 1ll << 26;

template <int BITS>
struct Cfg;
template <>
struct Cfg<2> {
  static constexpr int STAGES = 4;
  static constexpr int LUT_WORDS = 16 * 32;   // 4-bit pair index, replicated per lane
};
template <>
struct Cfg<4> {
  static constexpr int STAGES = 2;
  static constexpr int LUT_WORDS = 256;       // 8-bit pair index
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// bounded wait on an mbarrier phase; returns false if it gave up
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  uint32_t addr = smem_u32(bar);
  for (long long it = 0; it < WAIT_LIMIT; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// pair j of a lane chunk -> lut index
template <int BITS>
__device__ __forceinline__ uint32_t pair_index(const uint32_t *w, int j) {
  if (BITS == 2) return (w[j >> 3] >> (4 * (j & 7))) & 0xFu;
  return (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
}

template <int BITS>
__device__ __forceinline__ uint32_t lut_get(const uint32_t *lut, uint32_t idx, int lane) {
  if (BITS == 2) return lut[(idx << 5) | lane];
  return lut[idx];
}

// value tile: acc[mt] += Lcode[16 ch x 16 tok] * P[16 tok x 8 heads]
template <int BITS>
__device__ __forceinline__ void value_mma(float (&acc)[8][4], const uint32_t *vw, const uint32_t *vlut, int lane,
                                          uint32_t b0, uint32_t b1) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t A[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) A[r] = lut_get<BITS>(vlut, pair_index<BITS>(vw, 4 * mt + r), lane);
    mma16816(acc[mt], A, b0, b1);
  }
}

struct Merge {
  float m[WARPS][MAXGQ];
  float l[WARPS][MAXGQ];
  float o[WARPS][MAXM][MAXGQ][D];
};

template <int BITS, int G>
__global__ void __launch_bounds__(THREADS, 2) decode_kernel(const DecodeArgs a) {
  constexpr int STAGES = Cfg<BITS>::STAGES;
  constexpr int LANE_WORDS = BITS * 2;        // 32-bit words per lane chunk
  const PageLayout PL = page_layout(BITS, G);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;

  extern __shared__ __align__(128) unsigned char smem[];
  uint32_t *klut = reinterpret_cast<uint32_t *>(smem);
  uint32_t *vlut = klut + Cfg<BITS>::LUT_WORDS;
  float *qr = reinterpret_cast<float *>(vlut + Cfg<BITS>::LUT_WORDS);    // [8][128] stat order, scaled
  __half *qraw = reinterpret_cast<__half *>(qr + MAXGQ * D);             // [8][128] natural order
  uint64_t *bars = reinterpret_cast<uint64_t *>(qraw + MAXGQ * D);       // [WARPS][STAGES]
  unsigned char *stages = reinterpret_cast<unsigned char *>(bars + WARPS * STAGES);
  stages = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(stages) + 127) & ~uintptr_t(127));
  Merge &MG = *reinterpret_cast<Merge *>(stages);
  unsigned char *my_stage0 = stages + (size_t)warp * STAGES * PL.page_bytes;
  uint64_t *my_bars = bars + warp * STAGES;

  // code -> fp16 level tables (a pair of codes -> one half2)
  for (int i = tid; i < Cfg<BITS>::LUT_WORDS; i += THREADS) {
    uint32_t e = BITS == 2 ? (uint32_t)(i >> 5) : (uint32_t)i;
    uint32_t c0 = e & ((1u << BITS) - 1), c1 = e >> BITS;
    __half2 k2 = __halves2half2(a.klut_src[c0], a.klut_src[c1]);
    __half2 v2 = __halves2half2(a.vlut_src[c0], a.vlut_src[c1]);
    klut[i] = *reinterpret_cast<uint32_t *>(&k2);
    vlut[i] = *reinterpret_cast<uint32_t *>(&v2);
  }
  if (lane == 0)
    for (int s = 0; s < STAGES; ++s) mbar_init(&my_bars[s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  const int gq = a.Hq / a.Hkv;
  long long consumed = 0;                      // pages consumed by this warp so far (phase tracking)
  bool wait_failed = false;

  const int seg_begin = a.cta_seg[blockIdx.x], seg_end = a.cta_seg[blockIdx.x + 1];
  for (int seg = seg_begin; seg < seg_end; ++seg) {
    const int unit = a.segs[4 * seg + 0];
    const int pb = a.segs[4 * seg + 1], pe = a.segs[4 * seg + 2];
    const int session = unit / (a.L * a.Hkv);
    const int lh = unit % (a.L * a.Hkv);
    const int layer = lh / a.Hkv, kvh = lh % a.Hkv;
    const long long T = a.unit_len[unit];
    const long long Tf = (T / G) * G;
    const unsigned char *unit_pages = a.pages + (long long)unit * a.P_max * PL.page_bytes;

    // ---- rotate the query group once: q' = H (s o q) / d, in log2 units ----
    {
      const __half *qsrc = a.q + (((long long)session * a.L + layer) * a.Hq + (long long)kvh * gq) * D;
      for (int hh = warp; hh < MAXGQ; hh += WARPS) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int c = 4 * lane + j;
          __half hv = hh < gq ? qsrc[hh * D + c] : __float2half(0.f);
          qraw[hh * D + c] = hv;
          x[j] = __half2float(hv) * a.signs[c];
        }
        float y0 = x[0] + x[1], y1 = x[0] - x[1], y2 = x[2] + x[3], y3 = x[2] - x[3];
        x[0] = y0 + y2; x[2] = y0 - y2; x[1] = y1 + y3; x[3] = y1 - y3;
#pragma unroll
        for (int sm = 1; sm < 32; sm <<= 1) {
          const bool upper = (lane & sm) != 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float p = __shfl_xor_sync(FULL, x[j], sm);
            x[j] = upper ? p - x[j] : x[j] + p;
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int c = 4 * lane + j;
          int kb = c >> 4, r = c & 15;
          int pos = 32 * ((r & 7) >> 1) + 4 * kb + ((r & 1) | ((r >> 3) << 1));
          qr[hh * D + pos] = x[j] * (INV_D * LOG2E);
        }
      }
    }
    __syncthreads();

    // ---- per-warp state ----
    float acc[MAXM][8][4];
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[m][mt][r] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int npages = pe - pb;
    const int my_n = npages > warp ? (npages - warp + WARPS - 1) / WARPS : 0;
    // prologue
    if (lane == 0) {
      for (int k = 0; k < min(my_n, STAGES); ++k) {
        long long c = consumed + k;
        int st = (int)(c % STAGES);
        fence_async_smem();
        bulk_load(my_stage0 + (size_t)st * PL.page_bytes,
                  unit_pages + (long long)(pb + warp + k * WARPS) * PL.page_bytes, PL.page_bytes, &my_bars[st]);
      }
    }

    uint32_t bk[8][2];      // score B fragments of the current group (fp16 high part)
    uint32_t bl[8][2];      // and the fp16 residual
    float beta0 = 0.f, beta1 = 0.f;

    for (int k = 0; k < my_n; ++k) {
      const long long c = consumed + k;
      const int st = (int)(c % STAGES);
      const uint32_t par = (uint32_t)((c / STAGES) & 1);
      if (!mbar_wait(&my_bars[st], par)) {
        wait_failed = true;
        break;
      }
      __syncwarp();
      const unsigned char *sp = my_stage0 + (size_t)st * PL.page_bytes;
      const int page = pb + warp + k * WARPS;
      const long long tok0 = (long long)page * PAGE;
      const __half *norms = reinterpret_cast<const __half *>(sp + PL.off_norm);

#pragma unroll 1
      for (int tile = 0; tile < PAGE / TILE; ++tile) {
        const long long ts = tok0 + tile * TILE;
        if (ts >= T) break;
        float sc[4];
        if (ts < Tf) {
          if ((tile * TILE) % G == 0) {
            // new group: B = q' o (mx - mn) (fp16), beta = q' . mn
            const int gi = (tile * TILE) / G;
            const __half *st_mn = reinterpret_cast<const __half *>(sp + PL.off_stats + gi * 2 * D * 2);
            const __half *st_mx = st_mn + D;
            const float *qh = qr + g * D + 32 * t4;
            float bp = 0.f;
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
              const float4 qv = *reinterpret_cast<const float4 *>(qh + 4 * kb);
              const uint2 mnr = *reinterpret_cast<const uint2 *>(st_mn + 32 * t4 + 4 * kb);
              const uint2 mxr = *reinterpret_cast<const uint2 *>(st_mx + 32 * t4 + 4 * kb);
              const float2 mn01 = __half22float2(*reinterpret_cast<const __half2 *>(&mnr.x));
              const float2 mn23 = __half22float2(*reinterpret_cast<const __half2 *>(&mnr.y));
              const float2 mx01 = __half22float2(*reinterpret_cast<const __half2 *>(&mxr.x));
              const float2 mx23 = __half22float2(*reinterpret_cast<const __half2 *>(&mxr.y));
              const float a0 = qv.x * (mx01.x - mn01.x), a1 = qv.y * (mx01.y - mn01.y);
              const float a2 = qv.z * (mx23.x - mn23.x), a3 = qv.w * (mx23.y - mn23.y);
              bk[kb][0] = pack_h2(a0, a1);
              bk[kb][1] = pack_h2(a2, a3);
              // fp16 residuals: the score MMA runs on hi and lo so a keeps ~22 significant bits
              const float2 h01 = __half22float2(*reinterpret_cast<const __half2 *>(&bk[kb][0]));
              const float2 h23 = __half22float2(*reinterpret_cast<const __half2 *>(&bk[kb][1]));
              bl[kb][0] = pack_h2(a0 - h01.x, a1 - h01.y);
              bl[kb][1] = pack_h2(a2 - h23.x, a3 - h23.y);
              bp = fmaf(qv.x, mn01.x, bp);
              bp = fmaf(qv.y, mn01.y, bp);
              bp = fmaf(qv.z, mn23.x, bp);
              bp = fmaf(qv.w, mn23.y, bp);
            }
            bp += __shfl_xor_sync(FULL, bp, 1);
            bp += __shfl_xor_sync(FULL, bp, 2);
            beta0 = __shfl_sync(FULL, bp, 8 * t4);        // head 2*t4 lives in lanes 8*t4 .. +3
            beta1 = __shfl_sync(FULL, bp, 8 * t4 + 4);    // head 2*t4+1
          }
          uint32_t kw[LANE_WORDS];
#pragma unroll
          for (int i = 0; i < LANE_WORDS; i += 4) {
            const uint4 v4 = *reinterpret_cast<const uint4 *>(sp + tile * PL.tile_bytes + lane * PL.lane_bytes + 4 * i);
            kw[i] = v4.x; kw[i + 1] = v4.y; kw[i + 2] = v4.z; kw[i + 3] = v4.w;
          }
          sc[0] = beta0; sc[1] = beta1; sc[2] = beta0; sc[3] = beta1;
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            uint32_t A[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) A[r] = lut_get<BITS>(klut, pair_index<BITS>(kw, 4 * kb + r), lane);
            mma16816(sc, A, bk[kb][0], bk[kb][1]);
            mma16816(sc, A, bl[kb][0], bl[kb][1]);
          }
        } else {
          // trailing keys of an incomplete group: exact fp16 keys, unrotated query
          const __half *tail = a.tails + ((long long)a.unit_tail[unit] * a.units + unit) * (long long)G * D;
          const int r0 = (int)(ts - Tf) + g, r1 = r0 + 8;
          const int nt = (int)(T - Tf);
          sc[0] = sc[1] = sc[2] = sc[3] = 0.f;
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            const int c0 = 16 * kb + 2 * t4;
            uint32_t A[4];
            A[0] = r0 < nt ? *reinterpret_cast<const uint32_t *>(tail + r0 * D + c0) : 0u;
            A[1] = r1 < nt ? *reinterpret_cast<const uint32_t *>(tail + r1 * D + c0) : 0u;
            A[2] = r0 < nt ? *reinterpret_cast<const uint32_t *>(tail + r0 * D + c0 + 8) : 0u;
            A[3] = r1 < nt ? *reinterpret_cast<const uint32_t *>(tail + r1 * D + c0 + 8) : 0u;
            const uint32_t b0 = *reinterpret_cast<const uint32_t *>(qraw + g * D + c0);
            const uint32_t b1 = *reinterpret_cast<const uint32_t *>(qraw + g * D + c0 + 8);
            mma16816(sc, A, b0, b1);
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) sc[r] *= LOG2E * INV_SQRT_D;
        }
        // tokens past the end do not exist
        if (ts + g >= T) { sc[0] = -INFINITY; sc[1] = -INFINITY; }
        if (ts + g + 8 >= T) { sc[2] = -INFINITY; sc[3] = -INFINITY; }

        // ---- online softmax (base 2), heads 2*t4 and 2*t4+1 ----
        float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, o));
          x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, o));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        if (__any_sync(FULL, n0 > m0 || n1 > m1)) {
          const float s0 = ex2(m0 - n0), s1 = ex2(m1 - n1);
#pragma unroll
          for (int m = 0; m < MAXM; ++m)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              acc[m][mt][0] *= s0; acc[m][mt][2] *= s0;
              acc[m][mt][1] *= s1; acc[m][mt][3] *= s1;
            }
          l0 *= s0; l1 *= s1;
          m0 = n0; m1 = n1;
        }
        const float p0 = ex2(sc[0] - m0), p1 = ex2(sc[1] - m1);
        const float p2 = ex2(sc[2] - m0), p3 = ex2(sc[3] - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        const float na = ts + g < T ? __half2float(norms[tile * TILE + g]) : 0.f;
        const float nb = ts + g + 8 < T ? __half2float(norms[tile * TILE + g + 8]) : 0.f;

        uint32_t vw[LANE_WORDS];
#pragma unroll
        for (int i = 0; i < LANE_WORDS; i += 4) {
          const uint4 v4 =
              *reinterpret_cast<const uint4 *>(sp + PL.off_v + tile * PL.tile_bytes + lane * PL.lane_bytes + 4 * i);
          vw[i] = v4.x; vw[i + 1] = v4.y; vw[i + 2] = v4.z; vw[i + 3] = v4.w;
        }
        const uint32_t tmask = a.tmask[(long long)session * (a.cap / TILE) + ts / TILE];
        if (__popc(tmask) == 1) {
          const uint32_t b0 = transpose8x8(pack_h2(p0 * na, p1 * na));
          const uint32_t b1 = transpose8x8(pack_h2(p2 * nb, p3 * nb));
          const int m = __ffs(tmask) - 1;
          if (m == 0) value_mma<BITS>(acc[0], vw, vlut, lane, b0, b1);
          else if (m == 1) value_mma<BITS>(acc[1], vw, vlut, lane, b0, b1);
          else value_mma<BITS>(acc[2], vw, vlut, lane, b0, b1);
        } else {
          const uint8_t *modp = a.mod + (long long)session * a.cap + ts;
          const int ma = (ts + g < T) ? modp[g] : -1;
          const int mb = (ts + g + 8 < T) ? modp[g + 8] : -1;
#pragma unroll
          for (int m = 0; m < MAXM; ++m) {
            if (!(tmask & (1u << m))) continue;
            const float fa = ma == m ? na : 0.f, fb = mb == m ? nb : 0.f;
            const uint32_t b0 = transpose8x8(pack_h2(p0 * fa, p1 * fa));
            const uint32_t b1 = transpose8x8(pack_h2(p2 * fb, p3 * fb));
            value_mma<BITS>(acc[m], vw, vlut, lane, b0, b1);
          }
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
        for (long long c2 = consumed; c2 < consumed + min(my_n, STAGES); ++c2)
          (void)mbar_wait(&my_bars[c2 % STAGES], (uint32_t)((c2 / STAGES) & 1));
      return;
    }
    consumed += my_n;

    // ---- per-warp totals ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(FULL, l0, o);
      l1 += __shfl_xor_sync(FULL, l1, o);
    }
    __syncthreads();              // all warps done with their stage buffers
    if (g == 0) {
      MG.m[warp][2 * t4] = m0; MG.m[warp][2 * t4 + 1] = m1;
      MG.l[warp][2 * t4] = l0; MG.l[warp][2 * t4 + 1] = l1;
    }
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        MG.o[warp][m][2 * t4][16 * mt + g] = acc[m][mt][0];
        MG.o[warp][m][2 * t4 + 1][16 * mt + g] = acc[m][mt][1];
        MG.o[warp][m][2 * t4][16 * mt + g + 8] = acc[m][mt][2];
        MG.o[warp][m][2 * t4 + 1][16 * mt + g + 8] = acc[m][mt][3];
      }
    __syncthreads();
    float *part = a.partials + (long long)seg * MAXGQ * PARTIAL_FLOATS;
    for (int i = tid; i < MAXGQ * D; i += THREADS) {
      const int hh = i / D, ch = i % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) M = fmaxf(M, MG.m[w][hh]);
      float wsc[WARPS];
#pragma unroll
      for (int w = 0; w < WARPS; ++w) wsc[w] = MG.m[w][hh] == -INFINITY ? 0.f : ex2(MG.m[w][hh] - M);
      float *ph = part + hh * PARTIAL_FLOATS;
      if (ch == 0) {
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) L += wsc[w] * MG.l[w][hh];
        ph[0] = M;
        ph[1] = L;
      }
      for (int m = 0; m < a.M; ++m) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) o += wsc[w] * MG.o[w][m][hh][ch];
        ph[2 + m * D + ch] = o;
      }
    }
    __syncthreads();              // merge area is the stage ring of the next segment
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  __shared__ float Msh[MAXGQ], Lsh[MAXGQ];
  __shared__ float osh[MAXGQ][MAXM][D];
  const int unit = blockIdx.x, cb = blockIdx.y;
  const int tid = threadIdx.x;
  const int gq = a.Hq / a.Hkv;
  const int s0 = a.unit_seg[unit], s1 = a.unit_seg[unit + 1];
  if (tid < MAXGQ) {
    float M = -INFINITY, L = 0.f;
    for (int s = s0; s < s1; ++s) M = fmaxf(M, a.partials[((long long)s * MAXGQ + tid) * PARTIAL_FLOATS]);
    for (int s = s0; s < s1; ++s) {
      const float *p = a.partials + ((long long)s * MAXGQ + tid) * PARTIAL_FLOATS;
      if (p[0] != -INFINITY) L += ex2(p[0] - M) * p[1];
    }
    Msh[tid] = M;
    Lsh[tid] = L;
  }
  __syncthreads();
  for (int i = tid; i < MAXGQ * a.M * D; i += blockDim.x) {
    const int hh = i / (a.M * D), m = (i / D) % a.M, j = i % D;
    float o = 0.f;
    if (hh < gq) {
      for (int s = s0; s < s1; ++s) {
        const float *p = a.partials + ((long long)s * MAXGQ + hh) * PARTIAL_FLOATS;
        if (p[0] != -INFINITY) o += ex2(p[0] - Msh[hh]) * p[2 + m * D + j];
      }
    }
    osh[hh][m][j] = o;
  }
  __syncthreads();
  const int hh = tid >> 5, ci = cb * 32 + (tid & 31);
  const int session = unit / (a.L * a.Hkv);
  const int lh = unit % (a.L * a.Hkv);
  const int layer = lh / a.Hkv, kvh = lh % a.Hkv;
  if (hh < gq) {
    const float *R = a.rot + (long long)lh * a.M * D * D;
    float acc = 0.f;
    for (int m = 0; m < a.M; ++m)
      for (int j = 0; j < D; ++j) acc = fmaf(R[((long long)m * D + j) * D + ci], osh[hh][m][j], acc);
    const float L = Lsh[hh];
    const float y = L > 0.f ? acc / (L * 11.3137084989847603904f) : 0.f;
    a.out[(((long long)session * a.L + layer) * a.Hq + kvh * gq + hh) * D + ci] = __float2half_rn(y);
  }
}

template <int BITS, int G>
cudaError_t launch_decode_t(const DecodeArgs &a, int n_cta, cudaStream_t s) {
  static bool attr_done = false;
  const size_t smem = decode_smem_bytes(BITS, G);
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<BITS, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  decode_kernel<BITS, G><<<n_cta, THREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(int bits, int G) {
  const PageLayout PL = page_layout(bits, G);
  const int stages = bits == 2 ? Cfg<2>::STAGES : Cfg<4>::STAGES;
  const int lut = bits == 2 ? Cfg<2>::LUT_WORDS : Cfg<4>::LUT_WORDS;
  size_t head = 2 * lut * 4 + MAXGQ * D * 4 + MAXGQ * D * 2 + WARPS * stages * 8;
  size_t ring = (size_t)WARPS * stages * PL.page_bytes;
  if (ring < sizeof(Merge)) ring = sizeof(Merge);
  return head + 128 + ring;
}

cudaError_t launch_decode(const DecodeArgs &a, int n_cta, cudaStream_t s) {
  if (n_cta <= 0) return cudaSuccess;
  if (a.bits == 2 && a.G == 32) return launch_decode_t<2, 32>(a, n_cta, s);
  if (a.bits == 2 && a.G == 64) return launch_decode_t<2, 64>(a, n_cta, s);
  if (a.bits == 4 && a.G == 32) return launch_decode_t<4, 32>(a, n_cta, s);
  return launch_decode_t<4, 64>(a, n_cta, s);
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
  if (a.units <= 0) return cudaSuccess;
  dim3 grid((unsigned)a.units, D / 32);
  combine_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace okvq
