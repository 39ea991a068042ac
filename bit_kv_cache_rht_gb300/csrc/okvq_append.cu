// Append kernel: rotate + quantize + pack one chunk of tokens into the cache.
//
// "OmniKVQuant: KV Cache Quantization for Omni-LLMs", section 2 METHOD:
//   keys   - randomized Hadamard rotation (TurboQuant bullet), then min-max
//            scaling within each group of consecutive tokens with stored group
//            statistics and the shared fixed codebook (first OmniKVQuant bullet);
//   values - magnitude/direction split (TurboQuant bullet), rotation by the
//            token's modality eigenbasis (second OmniKVQuant bullet), the same
//            fixed codebook; everything bit-packed.
//
// One CTA per (touched 64-token page, layer, kv head). Values of the new tokens
// are quantized at once; a key group is quantized by the CTA whose page holds it
// when its last token arrives, reading earlier members from the fp16 tail buffer.
// The CTA owning the last touched page writes the new fp16 tail into the other
// tail buffer, so no CTA writes memory another CTA reads.
#include "okvq_internal.h"

namespace okvq {

namespace {

constexpr int THREADS = 256;
constexpr float INV_SQRT_D = 0.0883883476483184405501f;   // fp32(1/sqrt(128))
constexpr float SQRT_D = 11.3137084989847603904f;

constexpr int ROW_H = ROT_ROW_H;           // padded fp16 row: ldmatrix row reads hit distinct banks

// Shared memory of the value role: one part of R_m, the page's values, their codes.
struct ValueSmem {
  __half rh[D][ROW_H];             // one part (fp16 high, then residual) of R_m, [output][channel]
  __half vh[PAGE][ROW_H];          // the page's values, fp16 [token][channel]
  uint64_t bar;                    // completion of the bulk copy of rh
  uint8_t vc[PAGE * D];            // value codes of the page
  float vnorm[PAGE];
  int mod[PAGE];
  int present[MAXM];
};
// Shared memory of the key role: rotated keys, their codes and group statistics.
struct KeySmem {
  float xt[PAGE * D];              // keys [token][c] (rotated, fp32)
  uint8_t kc[PAGE * D];            // key codes of the page
  float kmn[2][D], kmx[2][D];     // group min and range (fp16 values held as fp32)
  float red[2][2][D];              // per-half min / max of a group
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// bounded wait on an mbarrier phase; false if it gave up
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity) {
  for (long long it = 0; it < (1ll << 26); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// code = number of thresholds strictly below x (NTHR = levels - 1)
template <int NTHR>
__device__ __forceinline__ int code_of(float x, const float *thr) {
  int c = 0;
#pragma unroll
  for (int j = 0; j < NTHR; ++j) c += x > thr[j] ? 1 : 0;
  return c;
}

// Canonical fp32 key rotation of one token, warp-wide: lane holds channels
// 4*lane .. 4*lane+3 of k' = fp32(1/sqrt d) * FWHT(s o k) (butterfly strides 1 and 2
// inside the lane, 4 .. 64 across lanes, round-to-nearest adds, no contraction).
__device__ __forceinline__ void rotate_key_row(uint2 raw, const float *signs, int lane, float (&x)[4]) {
  const __half2 h01 = *reinterpret_cast<const __half2 *>(&raw.x), h23 = *reinterpret_cast<const __half2 *>(&raw.y);
  x[0] = __low2float(h01) * signs[4 * lane];
  x[1] = __high2float(h01) * signs[4 * lane + 1];
  x[2] = __low2float(h23) * signs[4 * lane + 2];
  x[3] = __high2float(h23) * signs[4 * lane + 3];
  float y0 = __fadd_rn(x[0], x[1]), y1 = __fsub_rn(x[0], x[1]);
  float y2 = __fadd_rn(x[2], x[3]), y3 = __fsub_rn(x[2], x[3]);
  x[0] = __fadd_rn(y0, y2); x[2] = __fsub_rn(y0, y2);
  x[1] = __fadd_rn(y1, y3); x[3] = __fsub_rn(y1, y3);
#pragma unroll
  for (int sm = 1; sm < 32; sm <<= 1) {
    const bool upper = (lane & sm) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, x[j], sm);
      x[j] = upper ? __fsub_rn(p, x[j]) : __fadd_rn(x[j], p);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = __fmul_rn(x[j], INV_SQRT_D);
}

// Pack the codes of tile `tile` (16 tokens) from codes[64][128] into lane chunks.
// KIND 0 = K layout, 1 = V layout. Tokens >= valid_end (page-relative) pack as 0.
// The code slots of a word are unrolled, so their (token, channel) positions
// reduce to a few operations on the lane and word index.
template <int BITS, int KIND>
__device__ void pack_tile(const uint8_t *codes, uint8_t *dst, int tile, int valid_end, int tid, int nthreads) {
  constexpr int WPL = BITS * 2;                 // 32-bit words per lane chunk (16 B or 32 B)
  for (int w = tid; w < 32 * WPL; w += nthreads) {
    const int lane = w / WPL, wi = w % WPL;
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 32; b += BITS) {
      int j, e, tok, ch;
      chunk_code_at(KIND, BITS, wi, b, j, e);
      if (KIND == 0) k_pair_coords(lane, j, e, tok, ch);
      else v_pair_coords(lane, j, e, tok, ch);
      tok += 16 * tile;
      const uint32_t c = tok < valid_end ? codes[tok * D + ch] : 0u;
      word |= c << b;
    }
    reinterpret_cast<uint32_t *>(dst)[lane * WPL + wi] = word;
  }
}

// Inverse of pack_tile for tokens < keep_end (page-relative): fill codes[][] from dst.
template <int BITS, int KIND>
__device__ void unpack_tile(uint8_t *codes, const uint8_t *src, int tile, int keep_end, int tid, int nthreads) {
  constexpr int WPL = BITS * 2;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  for (int w = tid; w < 32 * WPL; w += nthreads) {
    const int lane = w / WPL, wi = w % WPL;
    const uint32_t word = reinterpret_cast<const uint32_t *>(src)[lane * WPL + wi];
#pragma unroll
    for (int b = 0; b < 32; b += BITS) {
      int j, e, tok, ch;
      chunk_code_at(KIND, BITS, wi, b, j, e);
      if (KIND == 0) k_pair_coords(lane, j, e, tok, ch);
      else v_pair_coords(lane, j, e, tok, ch);
      tok += 16 * tile;
      if (tok < keep_end) codes[tok * D + ch] = (uint8_t)((word >> b) & MASK);
    }
  }
}

// ROLE 0: the values of the new tokens (modality ids, norms, rotation, codes) and
// the page's tile masks; ROLE 1: the keys (groups that complete now, or every new
// token for TurboQuant keys) and the new fp16 tail. The two write disjoint parts of
// a page and read nothing the other writes, so they run as two concurrent grids.
template <int BITS, int ROLE>
__global__ void __launch_bounds__(THREADS) append_kernel(const AppendArgs a) {
  constexpr int NTHR = (1 << BITS) - 1;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PageLayout PL = page_layout(BITS, a.G);

  const long long page = a.page0 + blockIdx.x;
  const int lh = blockIdx.y;                       // layer * Hkv + kv head
  const long long unit = (long long)a.session * a.L * a.Hkv + lh;
  const long long P0 = page * PAGE;
  const long long T0 = a.T0, T1 = a.T0 + a.n;
  const int ta = (int)(max(P0, T0) - P0);          // new tokens [ta, tb) page-relative
  const int tb = (int)(min(P0 + PAGE, T1) - P0);
  const int row_stride = a.L * a.Hkv * D;          // between tokens in the input
  uint8_t *pg = a.pages + (unit * a.P_max + page) * (long long)PL.page_bytes;

  if constexpr (ROLE == 0) {
  ValueSmem &S = *reinterpret_cast<ValueSmem *>(smem_raw);
  // ---- modality ids of the new tokens (validated) ----
  for (int t = tid; t < PAGE; t += THREADS) {
    int m = 0;
    if (t >= ta && t < tb) {
      m = a.mod_in[P0 + t - T0];
      if (m >= a.M) {
        if (lh == 0) atomicOr(a.err, ERR_MODALITY);
        m = 0;
      }
    }
    S.mod[t] = m;
  }
  if (tid < MAXM) S.present[tid] = 0;
  __syncthreads();
  for (int t = ta + tid; t < tb; t += THREADS) S.present[S.mod[t]] = 1;
  if (lh == 0) {
    uint8_t *mod = a.mod + (long long)a.session * a.cap;
    for (int t = ta + tid; t < tb; t += THREADS) mod[P0 + t] = (uint8_t)S.mod[t];
  }
  // the page's own copy of its tile modality masks (decode reads them with the page)
  if (tid < PAGE / TILE) {
    const int t0 = tid * TILE, t1 = t0 + TILE;
    if (t1 > ta && t0 < tb) {
      uint8_t *tm = pg + PL.off_tmask + tid;
      uint8_t bitsm = (t0 < ta) ? *tm : 0;        // tile already partly filled
      for (int t = max(t0, ta); t < min(t1, tb); ++t) bitsm |= (uint8_t)(1u << S.mod[t]);
      *tm = bitsm;
    }
  }

  // ---- values: fp16 tile + norms ----
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&S.bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the new tokens' values: 8 tokens per warp, all loads issued first (lane: channels
  // 4 lane .. 4 lane + 3). Rows of other tokens are left as they are: a row only
  // feeds its own outputs, which are discarded.
  constexpr int VPW = PAGE / (THREADS / 32);
  uint2 vraw[VPW];
#pragma unroll
  for (int j = 0; j < VPW; ++j) {
    const int t = warp + j * (THREADS / 32);
    vraw[j] = make_uint2(0u, 0u);
    if (t >= ta && t < tb)
      vraw[j] = *reinterpret_cast<const uint2 *>(a.v + (P0 + t - T0) * (long long)row_stride + (long long)lh * D +
                                                 4 * lane);
  }
  // keep codes of older tokens that share a 16-token tile with the first new token
  if (ta % TILE != 0) unpack_tile<BITS, 1>(S.vc, pg + PL.off_v + (ta / TILE) * PL.tile_bytes, ta / TILE, ta, tid,
                                           THREADS);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < VPW; ++j) {
    const int t = warp + j * (THREADS / 32);
    if (t < ta || t >= tb) continue;               // warp-uniform
    *reinterpret_cast<uint2 *>(&S.vh[t][4 * lane]) = vraw[j];
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2 *>(&vraw[j].x));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2 *>(&vraw[j].y));
    float ss = x01.x * x01.x;
    ss = fmaf(x01.y, x01.y, ss);
    ss = fmaf(x23.x, x23.x, ss);
    ss = fmaf(x23.y, x23.y, ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float n = sqrtf(ss);
    if (lane == 0) {
      S.vnorm[t] = n;
      reinterpret_cast<__half *>(pg + PL.off_norm)[t] = __float2half_rn(n);
    }
  }
  __syncthreads();

  // ---- values: w = sqrt(d) * R_m v / |v| per modality present, then codes ----
  // On the tensor cores: [64 tokens x 128 ch] (fp16, exact) times R_m^T, with R_m in
  // fp16 high + residual parts (two MMAs, fp32 accumulation: ~2^-22 relative, as
  // fp32 arithmetic). Warp w: tokens 16 (w & 3) .., outputs 64 (w >> 2) ..
  const int mt = warp & 3, o0 = 64 * (warp >> 2);
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t phase = 0;
  bool failed = false;
  for (int m = 0; m < a.M && !failed; ++m) {
    if (!S.present[m]) continue;  // uniform: smem flag read after a barrier
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint32_t va = smem_addr(&S.vh[16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1)][8 * (lane >> 4)]);
    const int bj = lane >> 3;                      // ldmatrix matrix: output block (nt, nt + 1) x channel half
    const uint32_t rb = smem_addr(&S.rh[o0 + 8 * (bj >> 1) + (lane & 7)][8 * (bj & 1)]);
    // the high part, then the residual, staged in turn (one part of shared memory:
    // three CTAs fit on an SM); the products accumulate in fp32 across both passes
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {
      if (tid == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&S.bar)),
                     "r"((uint32_t)sizeof(S.rh))
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_addr(&S.rh[0][0])),
            "l"(a.rot_h + (((long long)lh * a.M + m) * 2 + part) * (D * ROW_H)), "r"((uint32_t)sizeof(S.rh)),
            "r"(smem_addr(&S.bar))
            : "memory");
      }
      failed = __syncthreads_or(!wait_bar(&S.bar, phase));
      phase ^= 1u;
      if (failed) {                                // the codes of this chunk's values stay unwritten
        if (tid == 0) atomicOr(a.err, ERR_WAIT);
        break;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t A[4];
        ldsm4(va + 32 * kk, A);
#pragma unroll
        for (int nt = 0; nt < 8; nt += 2) {
          uint32_t B[4];
          ldsm4(rb + (8 * nt * ROW_H) * 2 + 32 * kk, B);
          mma16816(acc[nt], A, B[0], B[1]);
          mma16816(acc[nt + 1], A, B[2], B[3]);
        }
      }
      __syncthreads();                             // rh is rewritten next
    }
    if (failed) break;
    // rows: tokens 16 mt + g (+8); columns: outputs o0 + 8 nt + 2 t4 (+1)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = 16 * mt + g + 8 * r;
      if (t >= ta && t < tb && S.mod[t] == m) {
        const float n = S.vnorm[t];
        const float sc = n > 0.f ? __fdiv_rn(SQRT_D, n) : 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int i = o0 + 8 * nt + 2 * t4;
          S.vc[t * D + i] = (uint8_t)code_of<NTHR>(acc[nt][2 * r] * sc, a.vthr);
          S.vc[t * D + i + 1] = (uint8_t)code_of<NTHR>(acc[nt][2 * r + 1] * sc, a.vthr);
        }
      }
    }
  }
  __syncthreads();                                 // every warp's codes are in S.vc
  // write the value tiles that got new tokens
  for (int tile = ta / TILE; tile * TILE < tb; ++tile)
    pack_tile<BITS, 1>(S.vc, pg + PL.off_v + tile * PL.tile_bytes, tile, tb, tid, THREADS);
  } else {
  KeySmem &S = *reinterpret_cast<KeySmem *>(smem_raw);
  if (a.G == 0) {
    // ---- TurboQuant keys (section 2, TurboQuant bullet): every new token now, like a
    // value with the shared Hadamard rotation: n = |k|, w = sqrt(d) k'/n, value levels ----
    // keep the codes of older tokens that share a 16-token tile with the first new token
    if (ta % TILE != 0) unpack_tile<BITS, 0>(S.kc, pg + (ta / TILE) * PL.tile_bytes, ta / TILE, ta, tid, THREADS);
    for (int t = ta + warp; t < tb; t += THREADS / 32) {
      const __half *src = a.k + (P0 + t - T0) * (long long)row_stride + (long long)lh * D;
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float v = __half2float(src[4 * lane + j]);
        ss = fmaf(v, v, ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float n = sqrtf(ss);
      float x[4];
      rotate_key_row(*reinterpret_cast<const uint2 *>(src + 4 * lane), a.signs, lane, x);
      const float sc = n > 0.f ? __fdiv_rn(SQRT_D, n) : 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) S.kc[t * D + 4 * lane + j] = (uint8_t)code_of<NTHR>(x[j] * sc, a.vthr);
      if (lane == 0) reinterpret_cast<__half *>(pg + PL.off_stats)[t] = __float2half_rn(n);
    }
    __syncthreads();
    for (int tile = ta / TILE; tile * TILE < tb; ++tile)
      pack_tile<BITS, 0>(S.kc, pg + tile * PL.tile_bytes, tile, tb, tid, THREADS);
    return;                       // no key groups, no fp16 tail
  }

  // ---- keys: groups that complete with this chunk, all of the page's at once ----
  const int G = a.G;
  float *xk = S.xt;               // keys as [token][c], row stride D
  uint32_t gmask = 0;             // bit gi: group gi of the page completes now
  for (int g0 = 0; g0 < PAGE; g0 += G) {
    const long long gend = P0 + g0 + G;
    if (gend > T0 && gend <= T1) gmask |= 1u << (g0 / G);
  }
  if (!gmask && blockIdx.x != gridDim.x - 1) return;   // nothing for this CTA
  if (gmask) {
    const __half *told = a.tail_old + unit * (long long)G * D;
    // rotate every member: warp per token (8 tokens per warp, loads issued first),
    // lane holds channels 4*lane .. 4*lane+3
    constexpr int PER_WARP = PAGE / (THREADS / 32);
    uint2 raw[PER_WARP];
#pragma unroll
    for (int j = 0; j < PER_WARP; ++j) {
      const int r = warp + j * (THREADS / 32);
      raw[j] = make_uint2(0u, 0u);
      if ((gmask >> (r / G)) & 1u) {
        const long long t = P0 + r, gs = P0 + (r / G) * G;
        const __half *src = t < T0 ? told + (t - gs) * D : a.k + (t - T0) * (long long)row_stride + (long long)lh * D;
        raw[j] = *reinterpret_cast<const uint2 *>(src + 4 * lane);
      }
    }
#pragma unroll
    for (int j = 0; j < PER_WARP; ++j) {
      const int r = warp + j * (THREADS / 32);
      if (!((gmask >> (r / G)) & 1u)) continue;     // warp-uniform
      float x[4];
      rotate_key_row(raw[j], a.signs, lane, x);
      *reinterpret_cast<float4 *>(&xk[r * D + 4 * lane]) = make_float4(x[0], x[1], x[2], x[3]);
    }
    __syncthreads();
    // per-channel statistics: thread (c, h) scans 32 members (G = 32: group h;
    // G = 64: half h of the group); then min rounded down, range rounded up
    {
      const int c = tid & (D - 1), h = tid / D;
      if ((gmask >> ((32 * h) / G)) & 1u) {
        float mn = xk[(32 * h) * D + c], mx = mn;
#pragma unroll 8
        for (int r = 1; r < 32; ++r) {
          const float v = xk[(32 * h + r) * D + c];
          mn = fminf(mn, v);
          mx = fmaxf(mx, v);
        }
        S.red[h][0][c] = mn;
        S.red[h][1][c] = mx;
      }
    }
    __syncthreads();
    for (int i = tid; i < (PAGE / G) * D; i += THREADS) {
      const int gi = i / D, c = i % D;
      if (!((gmask >> gi) & 1u)) continue;
      float mn, mx;
      if (G == 32) {
        mn = S.red[gi][0][c];
        mx = S.red[gi][1][c];
      } else {
        mn = fminf(S.red[0][0][c], S.red[1][0][c]);
        mx = fmaxf(S.red[0][1][c], S.red[1][1][c]);
      }
      const __half hmn = __float2half_rd(mn);
      const __half hrg = __float2half_ru(__fsub_ru(mx, __half2float(hmn)));
      S.kmn[gi][c] = __half2float(hmn);
      S.kmx[gi][c] = __half2float(hrg);
      __half *st = reinterpret_cast<__half *>(pg + PL.off_stats + gi * 2 * D * 2);
      st[stat_pos(c)] = hmn;
      st[D + stat_pos(c)] = hrg;
    }
    __syncthreads();
    {
      // thread (c, h): channel c of rows 32h .. 32h + 31, one group's statistics
      const int c = tid & (D - 1), h = tid / D, gi = (32 * h) / G;
      if ((gmask >> gi) & 1u) {
        const float mn = S.kmn[gi][c], rng = S.kmx[gi][c];
#pragma unroll 4
        for (int r = 32 * h; r < 32 * h + 32; ++r) {
          int code = 0;
          if (rng != 0.f) code = code_of<NTHR>(__fdiv_rn(__fsub_rn(xk[r * D + c], mn), rng), a.kthr);
          S.kc[r * D + c] = (uint8_t)code;
        }
      }
    }
    __syncthreads();
    for (int tile = 0; tile < PAGE / TILE; ++tile)
      if ((gmask >> ((TILE * tile) / G)) & 1u) pack_tile<BITS, 0>(S.kc, pg + tile * PL.tile_bytes, tile, PAGE, tid, THREADS);
    __syncthreads();
  }

  // ---- new fp16 tail (only the CTA of the last touched page) ----
  if (blockIdx.x == gridDim.x - 1) {
    long long tstart = (T1 / G) * G;
    const __half *told = a.tail_old + unit * (long long)G * D;
    __half *tnew = a.tail_new + unit * (long long)G * D;
    int ntail = (int)(T1 - tstart);
    for (int i = tid; i < ntail * D; i += THREADS) {
      int r = i / D, c = i % D;
      long long t = tstart + r;
      __half v = t < T0 ? told[(t - (T0 / G) * G) * D + c]
                        : a.k[(t - T0) * (long long)row_stride + (long long)lh * D + c];
      tnew[r * D + c] = v;
    }
  }
  }
}

template <int BITS, int ROLE>
cudaError_t set_append_attrs() {
  const int smem = ROLE == 0 ? (int)sizeof(ValueSmem) : (int)sizeof(KeySmem);
  cudaError_t r = cudaFuncSetAttribute(append_kernel<BITS, ROLE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(append_kernel<BITS, ROLE>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return r;
}

}  // namespace

// The value grid runs on `s`; the key grid on `aux`, forked from `s` before the
// value grid and joined back into `s` after it, so the two overlap on the device and
// everything issued on `s` afterwards sees both.
cudaError_t launch_append(const AppendArgs &a, int n_pages, cudaStream_t s, cudaStream_t aux, cudaEvent_t fork,
                          cudaEvent_t join) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] {
    cudaError_t r = set_append_attrs<2, 0>();
    if (r == cudaSuccess) r = set_append_attrs<2, 1>();
    if (r == cudaSuccess) r = set_append_attrs<4, 0>();
    if (r == cudaSuccess) r = set_append_attrs<4, 1>();
    return r;
  });
  if (e != cudaSuccess) return e;
  const dim3 grid(n_pages, a.L * a.Hkv);
  if ((e = cudaEventRecord(fork, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(aux, fork, 0)) != cudaSuccess) return e;
  if (a.bits == 2) append_kernel<2, 1><<<grid, THREADS, sizeof(KeySmem), aux>>>(a);
  else append_kernel<4, 1><<<grid, THREADS, sizeof(KeySmem), aux>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.bits == 2) append_kernel<2, 0><<<grid, THREADS, sizeof(ValueSmem), s>>>(a);
  else append_kernel<4, 0><<<grid, THREADS, sizeof(ValueSmem), s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaEventRecord(join, aux)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(s, join, 0);
}

}  // namespace okvq
