// Append kernels: rotate + quantize + pack one chunk of tokens into the cache.
//
// "OmniKVQuant: KV Cache Quantization for Omni-LLMs", section 2 METHOD:
//   keys   - randomized Hadamard rotation (TurboQuant bullet), then min-max
//            scaling within each group of consecutive tokens with stored group
//            statistics and the shared fixed codebook (first OmniKVQuant bullet);
//   values - magnitude/direction split (TurboQuant bullet), rotation by the
//            token's modality eigenbasis (second OmniKVQuant bullet), the same
//            fixed codebook; everything bit-packed.
//
// Two grids that write disjoint parts of the touched pages and read nothing the
// other writes, so they run concurrently:
//   append_value_kernel - one CTA per (run of touched pages, layer, kv head): the
//     modality ids, tile masks, value norms and value codes. Pages arrive by TMA
//     (128-byte swizzle) and R_m (fp16 high and residual parts) sits in tensor
//     memory; producer warps issue the 5th-generation MMAs D[128 outputs x 64
//     tokens] = R_m V^T and take the norms, consumer warps quantize the accumulator
//     (lane o = output channel o) and pack the codes straight into the decode's lane
//     chunks.
//   append_key_kernel - one CTA per (key group touched, layer, kv head): a group is
//     quantized when its last token arrives, earlier members read from the fp16 tail
//     buffer; the CTA of the last touched group writes the new fp16 tail into the
//     other tail buffer. append_turbo_kernel - TurboQuant keys (one CTA per touched
//     page): every new token coded on arrival.
#include <cuda.h>

#include "okvq_append.h"

namespace okvq {

namespace {

constexpr int THREADS = 256;                 // key kernel
constexpr float INV_SQRT_D = 0.0883883476483184405501f;   // fp32(1/sqrt(128))
constexpr float SQRT_D = 11.3137084989847603904f;

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

// ---------------------------------------------------------------------------
// Values: w = sqrt(d) R_m v / |v| on the 5th-generation tensor cores, then codes
// ---------------------------------------------------------------------------
constexpr int VWARPS = 8;                  // warp w reads accumulator lanes 32 (w % 4) .. (all 64 tokens when 4 warps)
constexpr int VTHREADS = 32 * VWARPS;
constexpr uint32_t V_TMEM_COLS = 256;      // two accumulators of 64 fp32 columns, then R_m (2 x 64 columns of fp16 pairs)
constexpr uint32_t V_TMEM_R = 128;         // first column of R_m: high part, then residual
constexpr int V_NBUF = 3;                  // pages in flight
constexpr int V_MAX_ROUNDS = V_MAX_PPC * MAXM;
constexpr int V_HALF_BYTES = PAGE * 64 * 2;    // one 64-channel half of a page: 64 rows of 128 B

// Shared memory of the value kernel (1024-byte aligned: the pages use the 128-byte
// swizzle, whose pattern repeats every 8 rows of 128 B).
struct ValueSmem {
  __half v[V_NBUF][PAGE * D];      // pages as the TMA writes them: two halves [64 tokens][64 channels], swizzled
  float sc[2][PAGE];               // sqrt(d) / |v| of a round's tokens (0: zero vector)
  uint8_t mod[V_MAX_PPC * PAGE];   // modality of each new token of the run, 0xff for the others
  uint8_t rpage[V_MAX_ROUNDS];     // rounds: (page of the run, modality)
  uint8_t rmod[V_MAX_ROUNDS];
  int pm[V_MAX_PPC];               // modalities present among a page's new tokens
  uint32_t mmask[2][2];            // a round's tokens
  int nround;
  uint32_t tmem;
  int mma_issued;                  // rounds whose MMAs were issued (producer thread 0)
  int pages_seen;                  // pages whose copy a producer saw complete
  uint64_t bar_v[V_NBUF], bar_mma[2];
  uint64_t bar_full[2], bar_empty[2], bar_rload;   // producer / consumer handshakes
};
constexpr size_t V_SMEM_BYTES = sizeof(ValueSmem) + 1024;   // + alignment slack

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand with the 128-byte swizzle:
// rows of 64 fp16 (128 B), 8-row groups 1024 B apart; a K step of 16 inside the
// 64-channel span advances the start by 32 B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// 32 consecutive 32-bit columns of this warp's 32 tensor-memory lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Bits of one V-layout chunk word (lane group t4) that belong to tokens below
// `keep_end` (tile-relative): the older tokens of a tile that a chunk extends.
template <int BITS>
__device__ __forceinline__ uint32_t v_keep_mask(int t4, int keep_end) {
  uint32_t m = 0;
#pragma unroll
  for (int jj = 0; jj < (BITS == 2 ? 8 : 4); ++jj)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tok = 2 * t4 + 8 * ((jj & 3) >> 1) + e;
      const int bit = BITS == 2 ? 4 * jj + 2 * e : 8 * jj + 4 * e;
      if (tok < keep_end) m |= ((1u << BITS) - 1u) << bit;
    }
  return m;
}

// One CTA per (run of a.vppc touched pages, layer * Hkv + kv head). Pages arrive by
// TMA (two 64-channel boxes each, 128-byte swizzle, three pages ahead); R_m sits in
// tensor memory (row o = lane o, fp16 pairs). A round is one (page, modality) pair:
// one thread issues D[o][t] = sum_c (R_hi[o][c] + R_lo[o][c]) v[t][c] (16 MMAs,
// M = 128, N = 64, K = 16, A from tensor memory, B from shared memory, fp32
// accumulation in tensor memory) and the round's norms are taken meanwhile. The
// MMAs of round r + 1 run while the warps quantize round r from the other
// accumulator: w = D[o][t] * sqrt(d) / |v_t| against the value thresholds.
//
// Packing: the thread of accumulator lane o = 32 quarter + 8 i + g holds channel o
// of its tokens; in the V layout channel o of decode lane (g, t4) sits in chunk
// word `quarter` (2-bit) or 2 quarter + i/2 (4-bit), at a bit offset set by i, the
// token's half and parity. The four (2-bit) or two (4-bit) threads that share a
// word are lanes g + 8 i of one warp, so two (one) xor-shuffles complete it.
// WIDE: the register budget of two value CTAs per SM beside the key CTAs (long
// chunks); otherwise one per SM, with the first part of R_m fetched whole at start.
template <int BITS, bool WIDE>
__global__ void __launch_bounds__(VTHREADS, WIDE ? 3 : 2)
    append_value_kernel(const AppendArgs a, const __grid_constant__ CUtensorMap tmv) {
  constexpr int PW = BITS / 2;                     // chunk words a thread stores per tile
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ValueSmem &S = *reinterpret_cast<ValueSmem *>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quarter = warp & 3, half = warp >> 2;
  const int gq = lane & 7, iq = lane >> 3;
  const PageLayout PL = page_layout(BITS, a.G);
  const int lh = blockIdx.y;
  const long long unit = (long long)a.session * a.L * a.Hkv + lh;
  const long long T0 = a.T0, T1 = a.T0 + a.n;
  const long long pbeg = a.page0 + (long long)blockIdx.x * a.vppc;
  const int npg = (int)(min(pbeg + a.vppc, (T1 - 1) / PAGE + 1) - pbeg);
  // one thread: page p of the run (all 64 rows; rows outside the input read as zeros)
  auto issue_page = [&](int p) {
    const int buf = p % V_NBUF;
    const int y = (int)((pbeg + p) * PAGE - T0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&S.bar_v[buf])),
                 "r"((uint32_t)(2 * V_HALF_BYTES))
                 : "memory");
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              smem_addr(&S.v[buf][0]) + (uint32_t)(h * V_HALF_BYTES)),
          "l"(reinterpret_cast<uint64_t>(&tmv)), "r"(lh * D + 64 * h), "r"(y), "r"(smem_addr(&S.bar_v[buf]))
          : "memory");
  };

  // R_m into tensor memory: warp w writes part w / 4 of rows 32 (w % 4) .. (row o =
  // lane o, fp16 pairs); every load of the row is issued before the stores
  const int rpart = half, rrow = 32 * quarter + lane;     // 8 warps: part w / 4; 4 warps: both parts in turn
  auto fetch_r = [&](int m, int part, int hh, uint4 (&rr)[8]) {   // half row hh of part `part`
    const uint4 *src = reinterpret_cast<const uint4 *>(a.rot_h + ((long long)(lh * a.M + m) * 2 + part) * D * D +
                                                       (long long)rrow * D) + 8 * hh;
#pragma unroll
    for (int k = 0; k < 8; ++k) rr[k] = src[k];
  };

  // the rotation of modality 0 (usually the first round's) is on its way during the
  // bookkeeping below
  constexpr int NPRE = WIDE ? 1 : 2;               // half rows of R_m fetched at kernel start
  uint4 rfirst[NPRE][8];
#pragma unroll
  for (int h = 0; h < NPRE; ++h) fetch_r(0, rpart, h, rfirst[h]);

  // ---- the run's modality ids (validated) and the session's copy of them; every
  // load issued before the first store ----
  {
    constexpr int PER = V_MAX_PPC * PAGE / VTHREADS;
    int mv[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const long long t = pbeg * PAGE + tid + k * VTHREADS;
      mv[k] = (tid + k * VTHREADS < npg * PAGE && t >= T0 && t < T1) ? (int)a.mod_in[t - T0] : 0xff;
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + k * VTHREADS;
      if (i >= npg * PAGE) break;
      int m = mv[k];
      if (m != 0xff) {
        if (m >= a.M) {
          if (lh == 0) atomicOr(a.err, ERR_MODALITY);
          m = 0;
        }
        if (lh == 0) a.mod[(long long)a.session * a.cap + pbeg * PAGE + i] = (uint8_t)m;
      }
      S.mod[i] = (uint8_t)m;
    }
  }
  if (tid < V_MAX_PPC) S.pm[tid] = 0;
  if (tid == 0) {
    for (int b = 0; b < V_NBUF; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&S.bar_v[b])));
    for (int b = 0; b < 2; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&S.bar_mma[b])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&S.bar_full[b])), "r"(VTHREADS / 2));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&S.bar_empty[b])), "r"(VTHREADS / 2));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&S.bar_rload)), "r"(VTHREADS / 2));
    S.mma_issued = 0;
    S.pages_seen = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int p = 0; p < V_NBUF && p < npg; ++p) issue_page(p);    // the first pages, before the bookkeeping
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                 "n"(V_TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem;
  auto store_r = [&](int part, int hh, const uint4 (&rr)[8]) {
    uint32_t r[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      r[4 * k] = rr[k].x;
      r[4 * k + 1] = rr[k].y;
      r[4 * k + 2] = rr[k].z;
      r[4 * k + 3] = rr[k].w;
    }
    tmem_st32(tmem + ((uint32_t)(32 * quarter) << 16) + V_TMEM_R + 64 * part + 32 * hh, r);
  };
  // R_m of modality m into tensor memory (this warp's parts, half rows in turn); the
  // first NPRE half rows may already be in `first`
  auto load_r = [&](int m, uint4 (&first)[NPRE][8], bool have_first) {
    for (int part = rpart; part < 2; part += VWARPS / 4)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint4 (&buf)[8] = first[hh % NPRE];
        if (!(have_first && part == rpart && hh < NPRE)) fetch_r(m, part, hh, buf);
        store_r(part, hh, buf);
      }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  };
  for (int i = tid; i < npg * PAGE; i += VTHREADS)
    if (S.mod[i] != 0xff) atomicOr(&S.pm[i / PAGE], 1 << S.mod[i]);
  __syncthreads();
  // ---- rounds: a page's modalities, the resident rotation's first, so that R_m is
  // copied again only when the modality changes ----
  if (tid == 0) {
    int n = 0, cur = -1;
    for (int p = 0; p < npg; ++p) {
      const int pm = S.pm[p];
      int done = 0;
      if (cur >= 0 && ((pm >> cur) & 1)) {
        S.rpage[n] = (uint8_t)p;
        S.rmod[n++] = (uint8_t)cur;
        done = 1 << cur;
      }
      for (int m = 0; m < a.M; ++m)
        if (((pm >> m) & 1) && !((done >> m) & 1)) {
          S.rpage[n] = (uint8_t)p;
          S.rmod[n++] = (uint8_t)m;
          cur = m;
        }
    }
    S.nround = n;
  }
  __syncthreads();
  const int nr = S.nround;

  // ---- warp roles. Producers (warps 4-7): wait for a round's page, issue its MMAs
  // into accumulator r % 2 (once the consumers freed it), take the round's token mask
  // and norms, signal `full`. Consumers (warps 0-3, one accumulator lane quarter each,
  // all 64 tokens): wait for `full` and the MMAs, make and pack the codes, free the
  // accumulator (`empty`), store a page's words after its last round and copy in the
  // page three ahead. Every handshake is an mbarrier with a bounded wait. ----
  constexpr int NR = VTHREADS / 2;                 // threads per role
  const bool producer = warp >= VWARPS / 2;
  int c_waited = 0, pages_issued = min(npg, V_NBUF);
  if (nr > 0) {
    load_r(S.rmod[0], rfirst, S.rmod[0] == 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (producer) {
    const int ptid = tid - NR;
    int reloads = 0;
    for (int r = 0; r < nr; ++r) {
      const int p = S.rpage[r], m = S.rmod[r], buf = p % V_NBUF;
      bool ok = true;
      if (r > 0 && m != S.rmod[r - 1]) {
        // a new rotation, written once the previous round's MMAs (its last readers) are done
        ok = __all_sync(0xffffffffu, wait_bar(&S.bar_mma[(r - 1) & 1], (uint32_t)((r - 1) >> 1) & 1u));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int part = 0; part < 2; ++part)
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            fetch_r(m, part, hh, rfirst[0]);
            store_r(part, hh, rfirst[0]);
          }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&S.bar_rload)) : "memory");
        ++reloads;
      }
      // every wait is taken by the whole warp (warp-uniform outcome: the .aligned
      // tensor-memory instructions need converged warps)
      ok = __all_sync(0xffffffffu, wait_bar(&S.bar_v[buf], (uint32_t)(p / V_NBUF) & 1u));
      if (ok && ptid == 0) S.pages_seen = max(S.pages_seen, p + 1);
      if (ok && r >= 2) ok = __all_sync(0xffffffffu, wait_bar(&S.bar_empty[r & 1], (uint32_t)((r >> 1) - 1) & 1u));
      if (ok && reloads) ok = __all_sync(0xffffffffu, wait_bar(&S.bar_rload, (uint32_t)(reloads - 1) & 1u));
      if (!ok) break;
      if (ptid == 0) {
        tc_fence_after();
        const uint32_t idesc = (1u << 4) | ((uint32_t)(PAGE >> 3) << 17) | ((uint32_t)(D >> 4) << 24);
        const uint32_t vb = smem_addr(&S.v[buf][0]);
        const uint32_t dt = tmem + (uint32_t)((r & 1) * PAGE);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t at = tmem + V_TMEM_R + (uint32_t)(64 * part + 8 * ks);
            const uint64_t bd = sw128_desc(vb + (uint32_t)((ks >> 2) * V_HALF_BYTES + (ks & 3) * 32));
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(dt),
                "r"(at), "l"(bd), "r"(idesc), "r"((part | ks) ? 1u : 0u));
          }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_addr(&S.bar_mma[r & 1]))
                     : "memory");
        S.mma_issued = r + 1;
      }
      // the round's tokens
      if (ptid < PAGE) {
        const uint32_t b = __ballot_sync(0xffffffffu, S.mod[p * PAGE + ptid] == m);
        if (lane == 0) S.mmask[r & 1][ptid >> 5] = b;
      }
      // norms: 2 threads per token (thread q: channels 64q .. 64q+63), partial sums of 4
      // channels combined in the order of a 32-lane xor-shuffle tree over lanes holding
      // channels 4l .. 4l+3 (level 16 across the token's two threads, 8 .. 1 inside)
      {
        const int t = ptid >> 1, q = ptid & 1;
        float s16[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = 8 * q + k;
          const uint4 u = *reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned char *>(&S.v[buf][0]) +
                                                            (c >> 3) * V_HALF_BYTES + t * 128 + (((c & 7) ^ (t & 7)) << 4));
          const float2 x0 = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
          const float2 x1 = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
          const float2 x2 = __half22float2(*reinterpret_cast<const __half2 *>(&u.z));
          const float2 x3 = __half22float2(*reinterpret_cast<const __half2 *>(&u.w));
          float s0 = x0.x * x0.x;
          s0 = fmaf(x0.y, x0.y, s0);
          s0 = fmaf(x1.x, x1.x, s0);
          s0 = fmaf(x1.y, x1.y, s0);
          float s1 = x2.x * x2.x;
          s1 = fmaf(x2.y, x2.y, s1);
          s1 = fmaf(x3.x, x3.x, s1);
          s1 = fmaf(x3.y, x3.y, s1);
          s16[2 * k] = s0;                         // partial 16q + 2k
          s16[2 * k + 1] = s1;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) s16[i] = __fadd_rn(s16[i], __shfl_xor_sync(0xffffffffu, s16[i], 1));   // l, l + 16
#pragma unroll
        for (int st = 8; st >= 1; st >>= 1)
#pragma unroll
          for (int i = 0; i < st; ++i) s16[i] = __fadd_rn(s16[i], s16[i + st]);
        if (q == 0 && S.mod[p * PAGE + t] == m) {
          const float n = sqrtf(s16[0]);
          S.sc[r & 1][t] = n > 0.f ? __fdiv_rn(SQRT_D, n) : 0.f;
          uint8_t *pg = a.pages + (unit * a.P_max + pbeg + p) * (long long)PL.page_bytes;
          reinterpret_cast<__half *>(pg + PL.off_norm)[t] = __float2half_rn(n);
        }
      }
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&S.bar_full[r & 1])) : "memory");
    }
  } else {
    uint32_t pw[4][PW];                            // chunk words of the page's four tiles (this lane quarter)
    for (int r = 0; r < nr; ++r) {
      const int p = S.rpage[r];
      const long long P0 = (pbeg + p) * PAGE;
      const int ta = (int)(max(P0, T0) - P0), tb = (int)(min(P0 + PAGE, T1) - P0);
      uint8_t *pg = a.pages + (unit * a.P_max + pbeg + p) * (long long)PL.page_bytes;
      if (!__all_sync(0xffffffffu, wait_bar(&S.bar_full[r & 1], (uint32_t)(r >> 1) & 1u))) break;
      if (!__all_sync(0xffffffffu, wait_bar(&S.bar_mma[r & 1], (uint32_t)(r >> 1) & 1u))) break;
      c_waited = r + 1;
      tc_fence_after();
      if (r == 0 || S.rpage[r - 1] != p) {
#pragma unroll
        for (int tl = 0; tl < 4; ++tl)
#pragma unroll
          for (int k = 0; k < PW; ++k) pw[tl][k] = 0u;
      }
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {             // tokens 32 hc .. 32 hc + 31 (tiles 2 hc, 2 hc + 1)
        float acc[32];
        tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)((r & 1) * PAGE + 32 * hc), acc);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const uint32_t mm = S.mmask[r & 1][hc];
        const float4 *scv = reinterpret_cast<const float4 *>(&S.sc[r & 1][32 * hc]);
        uint32_t wr[2][4];
#pragma unroll
        for (int tl = 0; tl < 2; ++tl)
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4) wr[tl][t4] = 0u;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 sc4 = scv[j4];
          const float scj[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * j4 + jj;
            const float x = acc[j] * scj[jj];
            uint32_t code;
            if constexpr (BITS == 2) {               // sorted thresholds: one compare picks the half
              const bool up = x > a.vthr[1];
              code = (up ? 2u : 0u) + (x > (up ? a.vthr[2] : a.vthr[0]) ? 1u : 0u);
            } else {
              code = (uint32_t)code_of<(1 << BITS) - 1>(x, a.vthr);
            }
            code &= 0u - ((mm >> j) & 1u);
            const int tt = j & 15;
            wr[j >> 4][(tt & 7) >> 1] |= code << (BITS == 2 ? 8 * (tt >> 3) + 2 * (tt & 1) : 16 * (tt >> 3) + 4 * (tt & 1));
          }
        }
        if constexpr (BITS == 2) {
          const int sh = 16 * (iq >> 1) + 4 * (iq & 1);
#pragma unroll
          for (int tl = 0; tl < 2; ++tl)
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              uint32_t w = wr[tl][t4] << sh;
              w |= __shfl_xor_sync(0xffffffffu, w, 8);
              w |= __shfl_xor_sync(0xffffffffu, w, 16);
              if (t4 == iq) pw[2 * hc + tl][0] |= w;
            }
        } else {
          const int sh = 8 * (iq & 1);
#pragma unroll
          for (int tl = 0; tl < 2; ++tl)
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              uint32_t w = wr[tl][t4] << sh;
              w |= __shfl_xor_sync(0xffffffffu, w, 8);
              if ((t4 >> 1) == (iq & 1)) pw[2 * hc + tl][t4 & 1] |= w;
            }
        }
      }
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&S.bar_empty[r & 1])) : "memory");
      // the page's last round: store its chunk words (older tokens of a tile kept), and
      // its buffer (MMAs done, norms taken) takes the page three ahead
      if (r + 1 == nr || S.rpage[r + 1] != p) {
#pragma unroll
        for (int tau = 0; tau < 4; ++tau) {
          if (TILE * tau + TILE <= ta || TILE * tau >= tb) continue;
          uint32_t *tw = reinterpret_cast<uint32_t *>(pg + PL.off_v + tau * PL.tile_bytes);
#pragma unroll
          for (int k = 0; k < PW; ++k) {
            const int t4 = BITS == 2 ? iq : 2 * (iq & 1) + k;
            uint32_t *dst =
                BITS == 2 ? tw + (4 * gq + t4) * 4 + quarter : tw + (4 * gq + t4) * 8 + 2 * quarter + (iq >> 1);
            uint32_t val = pw[tau][k];
            if (TILE * tau < ta) val |= *dst & v_keep_mask<BITS>(t4, ta - TILE * tau);
            *dst = val;
          }
        }
        if (tid == 0 && p + V_NBUF < npg) {
          issue_page(p + V_NBUF);
          pages_issued = p + V_NBUF + 1;
        }
      }
    }
  }
  const bool mine_failed = producer ? false : c_waited < nr;
  // a producer that stopped early leaves the consumers waiting: they give up too
  __syncthreads();
  // the pages' own copy of their tile modality masks (decode reads them with the page)
  for (int i = tid; i < npg * (PAGE / TILE); i += VTHREADS) {
    const int p = i / (PAGE / TILE), tile = i % (PAGE / TILE);
    const long long P0 = (pbeg + p) * PAGE;
    const int ta = (int)(max(P0, T0) - P0), tb = (int)(min(P0 + PAGE, T1) - P0);
    const int t0 = tile * TILE, t1 = t0 + TILE;
    if (t1 > ta && t0 < tb) {
      uint8_t *tm = a.pages + (unit * a.P_max + pbeg + p) * (long long)PL.page_bytes + PL.off_tmask + tile;
      uint8_t bitsm = (t0 < ta) ? *tm : 0;        // tile already partly filled
      for (int t = max(t0, ta); t < min(t1, tb); ++t) bitsm |= (uint8_t)(1u << S.mod[p * PAGE + t]);
      *tm = bitsm;
    }
  }
  if (tid == 0 && mine_failed) {
    atomicOr(a.err, ERR_WAIT);
    // MMAs still in flight: wait (bounded) before their accumulator columns are freed
    for (int r = c_waited; r < S.mma_issued; ++r) (void)wait_bar(&S.bar_mma[r & 1], (uint32_t)(r >> 1) & 1u);
    // pages still on their way
    for (int p = S.pages_seen; p < pages_issued; ++p)
      (void)wait_bar(&S.bar_v[p % V_NBUF], (uint32_t)(p / V_NBUF) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(V_TMEM_COLS));
}

// ---------------------------------------------------------------------------
// Keys: the groups that complete with this chunk (or every new token for
// TurboQuant keys), and the new fp16 tail
// ---------------------------------------------------------------------------
constexpr int XS = D + 4;                  // padded row (floats) of the rotated keys in shared memory

// Shared memory of the key kernel: rotated keys (or TurboQuant codes), and per
// (group, channel) the record [min, code thresholds on k' - min].
template <int BITS, int GT>
struct KeySmem {
  static constexpr int NREC = 1 << BITS;   // min + (levels - 1) thresholds
  static constexpr int RSLOT = D + 6;      // record slots: channel c at c + 2 (c / 32)
  float xt[GT * XS];               // rotated keys [token][channel ^ 16 (token / 8 % 2)], fp32
  float rec[RSLOT][NREC];
  float red[2][2][D];              // per-half min / max of a 64-token group
  uint32_t sgn[D / 2];             // Hadamard signs of channel pairs as fp16x2 sign bits
};
// Column of channel c in row r of KeySmem::xt: the rows 8 apart that one warp writes
// land in different banks.
__device__ __forceinline__ int xt_col(int c, int r) { return c ^ (16 * ((r >> 3) & 1)); }
// Record slot of channel c: the four channels 32 apart that one warp reads together
// sit in different banks.
__device__ __forceinline__ int rec_slot(int c) { return c + 2 * (c >> 5); }

// The smallest fp32 d >= 0 with fl(d / rng) > t (IEEE division, round to nearest
// even), +inf when no d qualifies (rng 0 or infinite: every code is 0). The quotient
// is non-decreasing in d, so d >= key_threshold(t, rng) <=> fl(d / rng) > t, and a
// code taken as the count of thresholds below d equals the count of midpoints
// below the correctly rounded scaled key. The start fl(t * rng) is within a few
// ulps of the answer; the walks are bounded.
__device__ float key_threshold(float t, float rng) {
  if (!(rng > 0.f) || isinf(rng)) return __int_as_float(0x7f800000);
  float d = fmaxf(__fmul_rn(t, rng), 0.f);
  for (int it = 0; it < 64 && !(__fdiv_rn(d, rng) > t); ++it) d = __int_as_float(__float_as_int(d) + 1);
  for (int it = 0; it < 64 && d > 0.f; ++it) {
    const float dp = __int_as_float(__float_as_int(d) - 1);
    if (!(__fdiv_rn(dp, rng) > t)) break;
    d = dp;
  }
  return d;
}

// Canonical fp32 rotation of one key, four threads per token: thread q holds
// channels 32q .. 32q+31 as 16 channel pairs; strides 1 .. 16 inside the thread,
// 32 and 64 across the token's threads (lanes q ^ 1, q ^ 2). Round-to-nearest
// adds and subtracts (a - b as fma(b, -1, a)), then one multiply by fp32(1/sqrt d):
// the same operations on the same operands as the warp-per-token form.
__device__ __forceinline__ void rotate_key_quarter(const uint4 (&raw)[4], const uint32_t *sgn, int q,
                                                   float2 (&x)[16]) {
  const float2 NEG1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t h = w[m] ^ sgn[16 * q + 4 * k + m];      // s o k on the fp16 pair (exact)
      x[4 * k + m] = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    }
  }
#pragma unroll
  for (int p = 0; p < 16; ++p) {                               // stride 1: the two halves of a pair
    const float a0 = x[p].x, b0 = x[p].y;
    x[p] = make_float2(__fadd_rn(a0, b0), __fsub_rn(a0, b0));
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)                             // strides 2 .. 16: pairs h apart
#pragma unroll
    for (int p = 0; p < 16; ++p)
      if (!(p & h)) {
        const float2 a0 = x[p], b0 = x[p + h];
        x[p] = __fadd2_rn(a0, b0);
        x[p + h] = __ffma2_rn(b0, NEG1, a0);
      }
#pragma unroll
  for (int sm = 1; sm <= 2; sm <<= 1) {                        // strides 32, 64: partner lane q ^ sm
    const float s = (q & sm) ? -1.f : 1.f;                     // upper: partner - own, lower: own + partner
    const float2 s2 = make_float2(s, s);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, x[p].x, sm), __shfl_xor_sync(0xffffffffu, x[p].y, sm));
      x[p] = __ffma2_rn(s2, x[p], o);
    }
  }
  const float2 sc = make_float2(INV_SQRT_D, INV_SQRT_D);
#pragma unroll
  for (int p = 0; p < 16; ++p) x[p] = __fmul2_rn(x[p], sc);
}

// TurboQuant keys (section 2, TurboQuant bullet): every new token now, like a value
// with the shared Hadamard rotation: n = |k|, w = sqrt(d) k'/n, value levels. One CTA
// per (touched page, layer * Hkv + kv head); no groups, no fp16 tail.
struct TurboSmem {
  uint8_t kc[PAGE * D];            // key codes [token][channel]
};
template <int BITS>
__global__ void __launch_bounds__(THREADS) append_turbo_kernel(const AppendArgs a) {
  constexpr int NTHR = (1 << BITS) - 1;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PageLayout PL = page_layout(BITS, 0);
  const long long page = a.page0 + blockIdx.x;
  const int lh = blockIdx.y;                       // layer * Hkv + kv head
  const long long unit = (long long)a.session * a.L * a.Hkv + lh;
  const long long P0 = page * PAGE;
  const long long T0 = a.T0, T1 = a.T0 + a.n;
  const int ta = (int)(max(P0, T0) - P0);          // new tokens [ta, tb) page-relative
  const int tb = (int)(min(P0 + PAGE, T1) - P0);
  const int row_stride = a.L * a.Hkv * D;          // between tokens in the input
  uint8_t *pg = a.pages + (unit * a.P_max + page) * (long long)PL.page_bytes;
  TurboSmem &S = *reinterpret_cast<TurboSmem *>(smem_raw);
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
}

// Grouped keys: one CTA per (key group touched by the chunk, layer * Hkv + kv head),
// GT = group size tokens, 4 threads per token. A group is quantized when its last
// token arrives, earlier members read from the fp16 tail buffer; the CTA of the last
// touched group writes the new fp16 tail into the other tail buffer.
template <int BITS, int GT>
__global__ void __launch_bounds__(4 * GT) append_key_kernel(const AppendArgs a) {
  constexpr int NTHR = (1 << BITS) - 1;
  constexpr int NT = 4 * GT;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  KeySmem<BITS, GT> &S = *reinterpret_cast<KeySmem<BITS, GT> *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PageLayout PL = page_layout(BITS, GT);
  const long long T0 = a.T0, T1 = a.T0 + a.n;
  const long long gs = (T0 / GT + blockIdx.x) * GT;         // the group: tokens [gs, gs + GT)
  const int lh = blockIdx.y;                                 // layer * Hkv + kv head
  const long long unit = (long long)a.session * a.L * a.Hkv + lh;
  const long long page = gs / PAGE;
  const int g0 = (int)(gs - page * PAGE);                    // the group's first token in its page
  const int row_stride = a.L * a.Hkv * D;                    // between tokens in the input
  uint8_t *pg = a.pages + (unit * a.P_max + page) * (long long)PL.page_bytes;
  const __half *told = a.tail_old + unit * (long long)GT * D;

  if (gs + GT <= T1) {                                       // the group completes now
    if (tid < D / 2)
      S.sgn[tid] = (a.signs[2 * tid] < 0.f ? 0x8000u : 0u) | (a.signs[2 * tid + 1] < 0.f ? 0x80000000u : 0u);
    __syncthreads();
    // rotate every member: thread q of a token holds channels 32q .. 32q+31; warp w
    // takes tokens g = 4 (w % 2) .. + 3 and g + 8 of the group's tile w / 2
    const int q = lane & 3, tk = lane >> 4;
    const int tile = warp >> 1, g = 4 * (warp & 1) + ((lane >> 2) & 3);
    const int r = TILE * tile + g + 8 * tk;
    float2 x[16];
    {
      const long long t = gs + r;
      const __half *src = (t < T0 ? told + (t - gs) * D : a.k + (t - T0) * (long long)row_stride + (long long)lh * D) +
                          32 * q;
      uint4 raw[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) raw[k] = reinterpret_cast<const uint4 *>(src)[k];
      rotate_key_quarter(raw, S.sgn, q, x);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4 *>(&S.xt[r * XS + xt_col(32 * q + 4 * k, r)]) =
            make_float4(x[2 * k].x, x[2 * k].y, x[2 * k + 1].x, x[2 * k + 1].y);
    }
    __syncthreads();
    // per-channel statistics: thread (c, h) scans members 32h .. 32h + 31
    {
      const int c = tid & (D - 1), h = tid / D;
      float mn = S.xt[(32 * h) * XS + xt_col(c, 0)], mx = mn;
#pragma unroll 8
      for (int rr = 1; rr < 32; ++rr) {
        const float v = S.xt[(32 * h + rr) * XS + xt_col(c, rr)];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
      S.red[h][0][c] = mn;
      S.red[h][1][c] = mx;
    }
    __syncthreads();
    // min rounded down, range rounded up (fp16, stored), and the code thresholds
    if (tid < D) {
      const int c = tid;
      float mn = S.red[0][0][c], mx = S.red[0][1][c];
      if (GT == 64) {
        mn = fminf(mn, S.red[1][0][c]);
        mx = fmaxf(mx, S.red[1][1][c]);
      }
      const __half hmn = __float2half_rd(mn);
      const __half hrg = __float2half_ru(__fsub_ru(mx, __half2float(hmn)));
      __half *st = reinterpret_cast<__half *>(pg + PL.off_stats + (g0 / GT) * 2 * D * 2);
      st[stat_pos(c)] = hmn;
      st[D + stat_pos(c)] = hrg;
      const float rng = __half2float(hrg);
      float *rec = S.rec[rec_slot(c)];
      rec[0] = __half2float(hmn);
#pragma unroll
      for (int j = 0; j < NTHR; ++j) rec[1 + j] = key_threshold(a.kthr[j], rng);
    }
    __syncthreads();
    // codes from the registers, straight into chunk words (k_pair_coords, k_code_bit):
    // channel 32q + i of token g + 8 tk goes to decode lane (g, t4) at
    //   2-bit: word q,           i = 2 t4 + e + 8 s + 16 hb, bit 8 (2 hb + tk) + 4 s + 2 e
    //   4-bit: word 2q + i / 16, i = 2 t4 + e + 8 s + 16 hb, bit 8 (2 s + tk) + 4 e
    // and the partner token (tk ^ 1) is lane ^ 16.
    uint32_t pw[2][4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) pw[hh][t4] = 0u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float4 *rv = reinterpret_cast<const float4 *>(S.rec[rec_slot(32 * q + i)]);
      const float4 r0 = rv[0];
      const float xv = (i & 1) ? x[i >> 1].y : x[i >> 1].x;
      const float dm = __fsub_rn(xv, r0.x);
      uint32_t code = (dm >= r0.y) + (dm >= r0.z) + (dm >= r0.w);
      if constexpr (BITS == 4) {
#pragma unroll
        for (int kk = 1; kk < 4; ++kk) {
          const float4 rk = rv[kk];
          code += (dm >= rk.x) + (dm >= rk.y) + (dm >= rk.z) + (dm >= rk.w);
        }
      }
      const int e = i & 1, t4 = (i >> 1) & 3, sb = (i >> 3) & 1, hb = i >> 4;
      if (BITS == 2) pw[0][t4] |= code << (16 * hb + 4 * sb + 2 * e);
      else pw[hb][t4] |= code << (16 * sb + 4 * e);
    }
    uint32_t *tw = reinterpret_cast<uint32_t *>(pg + (g0 / TILE + tile) * PL.tile_bytes);
#pragma unroll
    for (int hh = 0; hh < BITS / 2; ++hh)
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) {
        uint32_t w = pw[hh][t4] << (8 * tk);
        w |= __shfl_xor_sync(0xffffffffu, w, 16);
        if ((t4 >> 1) == tk) {
          if (BITS == 2) tw[(4 * g + t4) * 4 + q] = w;
          else tw[(4 * g + t4) * 8 + 2 * q + hh] = w;
        }
      }
  }

  // ---- new fp16 tail (only the CTA of the last touched group): 16-byte pieces, every
  // load issued before the first store ----
  if (blockIdx.x == gridDim.x - 1) {
    const long long tstart = (T1 / GT) * GT, ts0 = (T0 / GT) * GT;
    __half *tnew = a.tail_new + unit * (long long)GT * D;
    const int npc = (int)(T1 - tstart) * (D / 8);
    constexpr int PER = (GT * (D / 8) + NT - 1) / NT;
    uint4 v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + k * NT;
      if (i < npc) {
        const long long t = tstart + (i >> 4);
        const int c = 8 * (i & 15);
        v[k] = *reinterpret_cast<const uint4 *>(t < T0 ? told + (t - ts0) * D + c
                                                       : a.k + (t - T0) * (long long)row_stride + (long long)lh * D + c);
      }
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + k * NT;
      if (i < npc) *reinterpret_cast<uint4 *>(tnew + (i >> 4) * D + 8 * (i & 15)) = v[k];
    }
  }
}

// Shared-memory sizes, and one carveout (all shared) for every append kernel: CTAs of
// kernels whose L1 / shared split differs do not share an SM, and the key CTAs are
// meant to run beside the value CTAs.
template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (r == cudaSuccess)
    r = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  return r;
}
template <int BITS>
cudaError_t set_append_attrs() {
  cudaError_t r = set_smem(append_value_kernel<BITS, false>, V_SMEM_BYTES);
  if (r == cudaSuccess) r = set_smem(append_value_kernel<BITS, true>, V_SMEM_BYTES);
  if (r == cudaSuccess) r = set_smem(append_key_kernel<BITS, 32>, sizeof(KeySmem<BITS, 32>));
  if (r == cudaSuccess) r = set_smem(append_key_kernel<BITS, 64>, sizeof(KeySmem<BITS, 64>));
  if (r == cudaSuccess) r = set_smem(append_turbo_kernel<BITS>, sizeof(TurboSmem));
  return r;
}

// cuTensorMapEncodeTiled, looked up in the driver once
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

}  // namespace

// The value grid runs on `s`; the key grid on `aux`, forked from `s` before the
// value grid and joined back into `s` after it, so the two overlap on the device and
// everything issued on `s` afterwards sees both.
cudaError_t launch_append(const AppendArgs &a, int n_pages, cudaStream_t s, cudaStream_t aux, cudaEvent_t fork,
                          cudaEvent_t join) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] {
    cudaError_t r = set_append_attrs<2>();
    if (r == cudaSuccess) r = set_append_attrs<4>();
    return r;
  });
  if (e != cudaSuccess) return e;
  if (a.vppc < 1 || a.vppc > V_MAX_PPC) return cudaErrorInvalidValue;
  // the chunk's values as a 2-D tensor [n tokens][L * Hkv * 128 channels]; a box is
  // 64 channels x 64 tokens, written to shared memory with the 128-byte swizzle
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmv;
  const cuuint64_t dims[2] = {(cuuint64_t)a.L * a.Hkv * D, (cuuint64_t)a.n};
  const cuuint64_t strides[1] = {(cuuint64_t)a.L * a.Hkv * D * sizeof(__half)};
  const cuuint32_t box[2] = {64, PAGE}, estr[2] = {1, 1};
  if (enc(&tmv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(a.v), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int upl = a.L * a.Hkv;
  const dim3 vgrid((n_pages + a.vppc - 1) / a.vppc, upl);
  // the value grid first (about one CTA per SM), then the key grid on `aux` fills the
  // room the value CTAs leave
  if ((e = cudaEventRecord(fork, s)) != cudaSuccess) return e;
  if (a.bits == 2) {
    if (a.vwide) append_value_kernel<2, true><<<vgrid, VTHREADS, V_SMEM_BYTES, s>>>(a, tmv);
    else append_value_kernel<2, false><<<vgrid, VTHREADS, V_SMEM_BYTES, s>>>(a, tmv);
  } else {
    if (a.vwide) append_value_kernel<4, true><<<vgrid, VTHREADS, V_SMEM_BYTES, s>>>(a, tmv);
    else append_value_kernel<4, false><<<vgrid, VTHREADS, V_SMEM_BYTES, s>>>(a, tmv);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(aux, fork, 0)) != cudaSuccess) return e;
  if (a.G == 0) {
    const dim3 tgrid(n_pages, upl);
    if (a.bits == 2) append_turbo_kernel<2><<<tgrid, THREADS, sizeof(TurboSmem), aux>>>(a);
    else append_turbo_kernel<4><<<tgrid, THREADS, sizeof(TurboSmem), aux>>>(a);
  } else {
    const long long T1 = a.T0 + a.n;
    const dim3 kgrid((unsigned)((T1 - 1) / a.G - a.T0 / a.G + 1), upl);
    if (a.G == 32) {
      if (a.bits == 2) append_key_kernel<2, 32><<<kgrid, 128, sizeof(KeySmem<2, 32>), aux>>>(a);
      else append_key_kernel<4, 32><<<kgrid, 128, sizeof(KeySmem<4, 32>), aux>>>(a);
    } else {
      if (a.bits == 2) append_key_kernel<2, 64><<<kgrid, 256, sizeof(KeySmem<2, 64>), aux>>>(a);
      else append_key_kernel<4, 64><<<kgrid, 256, sizeof(KeySmem<4, 64>), aux>>>(a);
    }
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaEventRecord(join, aux)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(s, join, 0);
}

}  // namespace okvq
