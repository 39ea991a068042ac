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
//     modality ids, tile masks, value norms and value codes. R_m (fp16 high and
//     residual parts) and the page's values sit in shared memory in the tensor
//     core's layout; one thread issues the 5th-generation MMAs
//     D[128 outputs x 64 tokens] = R_m V^T into tensor memory, and the thread of
//     output lane o quantizes its row and packs the codes straight into the
//     decode's lane chunks (the accumulator's lane/column order is the chunk's).
//   append_key_kernel - one CTA per (touched page, layer, kv head): a key group is
//     quantized by the CTA whose page holds it when its last token arrives,
//     reading earlier members from the fp16 tail buffer; the CTA owning the last
//     touched page writes the new fp16 tail into the other tail buffer.
#include "okvq_internal.h"

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
constexpr int VTHREADS = 128;              // epilogue: thread o = output channel o = tensor-memory lane o
constexpr uint32_t V_TMEM_COLS = 64;       // the accumulator: one fp32 column per token of a page
constexpr int V_MAX_ROUNDS = V_MAX_PPC * MAXM;

// Shared memory of the value kernel. R_m and a page's values use the K-major
// layout without swizzle (kmajor_off): core matrices of 8 rows x 8 channels.
struct ValueSmem {
  __half r[2][D * D];              // R_m, fp16 high part then residual; rows = output channels
  __half v[2][PAGE * D];           // values of a page (two buffers); rows = tokens
  float sc[PAGE];                  // sqrt(d) / |v| of the current round's tokens (0: zero vector)
  uint8_t mod[V_MAX_PPC * PAGE];   // modality of each new token of the run, 0xff for the others
  uint8_t rpage[V_MAX_ROUNDS];     // rounds: (page of the run, modality)
  uint8_t rmod[V_MAX_ROUNDS];
  int pm[V_MAX_PPC];               // modalities present among a page's new tokens
  uint32_t mmask[2];               // tokens of the current round
  int nround;
  uint32_t tmem;
  uint64_t bar_r, bar_mma;
};

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Shared-memory matrix descriptor of a K-major operand without swizzle: core
// matrices adjacent along K 128 B apart, along M/N 2 KB apart (kmajor_off).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(2048u >> 4) << 32) |
         (1ull << 46);
}

// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes
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

// One CTA per (run of a.vppc touched pages, layer * Hkv + kv head). A round is one
// (page, modality) pair: the page's new tokens of that modality are copied into
// shared memory (the next round's while this one computes), their norms taken,
// and one thread issues D[o][t] = sum_c (R_hi[o][c] + R_lo[o][c]) v[t][c] (16 MMAs,
// M = 128, N = 64, K = 16, fp32 accumulation in tensor memory). The thread of
// lane o then quantizes w = D[o][t] * sqrt(d) / |v_t| for the round's tokens.
//
// Packing: thread o = 32 w + 8 i + g holds channel o of every token; in the V
// layout channel o of decode lane (g, t4) sits in chunk word w (2-bit) or
// 2 w + i/2 (4-bit), at a bit offset set by i, the token's half and parity. The
// four (2-bit) or two (4-bit) threads that share a word are lanes g + 8 i of one
// warp, so two (one) xor-shuffles complete it.
template <int BITS>
__global__ void __launch_bounds__(VTHREADS, 2) append_value_kernel(const AppendArgs a) {
  constexpr int NTHR = (1 << BITS) - 1;
  constexpr int PW = BITS / 2;                     // chunk words a thread stores per tile
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ValueSmem &S = *reinterpret_cast<ValueSmem *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane & 7, iq = lane >> 3;
  const PageLayout PL = page_layout(BITS, a.G);
  const int lh = blockIdx.y;
  const long long unit = (long long)a.session * a.L * a.Hkv + lh;
  const long long T0 = a.T0, T1 = a.T0 + a.n;
  const long long pbeg = a.page0 + (long long)blockIdx.x * a.vppc;
  const int npg = (int)(min(pbeg + a.vppc, (T1 - 1) / PAGE + 1) - pbeg);
  const long long row_stride = (long long)a.L * a.Hkv * D;

  // ---- the run's modality ids (validated) and the session's copy of them ----
  for (int i = tid; i < npg * PAGE; i += VTHREADS) {
    const long long t = pbeg * PAGE + i;
    int m = 0xff;
    if (t >= T0 && t < T1) {
      m = a.mod_in[t - T0];
      if (m >= a.M) {
        if (lh == 0) atomicOr(a.err, ERR_MODALITY);
        m = 0;
      }
      if (lh == 0) a.mod[(long long)a.session * a.cap + t] = (uint8_t)m;
    }
    S.mod[i] = (uint8_t)m;
  }
  if (tid < V_MAX_PPC) S.pm[tid] = 0;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&S.bar_r)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&S.bar_mma)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
  for (int i = tid; i < npg * PAGE; i += VTHREADS)
    if (S.mod[i] != 0xff) atomicOr(&S.pm[i / PAGE], 1 << S.mod[i]);
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

  auto issue_r = [&](int m) {                      // one thread: both parts of R_m, one bulk copy
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&S.bar_r)),
                 "r"((uint32_t)sizeof(S.r))
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(&S.r[0][0])),
        "l"(a.rot_h + (long long)(lh * a.M + m) * 2 * D * D), "r"((uint32_t)sizeof(S.r)), "r"(smem_addr(&S.bar_r))
        : "memory");
  };
  auto issue_v = [&](int r, int buf) {             // every thread: the round's tokens, 16-byte copies
    const int p = S.rpage[r], m = S.rmod[r];
    const long long P0 = (pbeg + p) * PAGE;
    for (int i = tid; i < PAGE * (D / 8); i += VTHREADS) {
      const int t = i & (PAGE - 1), c = i >> 6;    // a warp: 32 tokens, one 8-channel block
      if (S.mod[p * PAGE + t] == m)
        cp_async16(&S.v[buf][kmajor_off(t, 8 * c)], a.v + (P0 + t - T0) * row_stride + (long long)lh * D + 8 * c);
    }
    cp_async_commit();
  };

  uint32_t ph_r = 0, ph_mma = 0;
  bool failed = false, r_pending = false, mma_pending = false;
  uint32_t pw[4][PW];
  if (nr > 0) {
    if (tid == 0) issue_r(S.rmod[0]);
    r_pending = true;
    issue_v(0, 0);
  }
  for (int r = 0; r < nr; ++r) {
    const int buf = r & 1, p = S.rpage[r], m = S.rmod[r];
    const long long P0 = (pbeg + p) * PAGE;
    const int ta = (int)(max(P0, T0) - P0), tb = (int)(min(P0 + PAGE, T1) - P0);
    uint8_t *pg = a.pages + (unit * a.P_max + pbeg + p) * (long long)PL.page_bytes;
    if (r == 0 || S.rpage[r - 1] != p) {
#pragma unroll
      for (int tau = 0; tau < 4; ++tau)
#pragma unroll
        for (int k = 0; k < PW; ++k) pw[tau][k] = 0u;
    }
    // the next round's values go to the other buffer (its MMA has completed)
    if (r + 1 < nr) {
      issue_v(r + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    if (warp < 2) {
      const uint32_t b = __ballot_sync(0xffffffffu, S.mod[p * PAGE + tid] == m);
      if (lane == 0) S.mmask[warp] = b;
    }
    __syncthreads();                               // the round's values (every thread's copies) landed
    // norms: thread t = token t, partial sums of 4 channels combined in the order of a
    // 32-lane xor-shuffle tree (lane l holding channels 4l .. 4l+3)
    if (tid < PAGE && S.mod[p * PAGE + tid] == m) {
      float q[32];
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(&S.v[buf][kmajor_off(tid, 8 * c)]);
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
        q[2 * c] = s0;
        q[2 * c + 1] = s1;
      }
#pragma unroll
      for (int s = 16; s >= 1; s >>= 1)
#pragma unroll
        for (int l = 0; l < s; ++l) q[l] = __fadd_rn(q[l], q[l + s]);
      const float n = sqrtf(q[0]);
      S.sc[tid] = n > 0.f ? __fdiv_rn(SQRT_D, n) : 0.f;
      reinterpret_cast<__half *>(pg + PL.off_norm)[tid] = __float2half_rn(n);
    }
    bool ok = true;
    if (r_pending) {                               // R_m resident
      ok = wait_bar(&S.bar_r, ph_r);
      if (ok) {
        ph_r ^= 1u;
        r_pending = false;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the copied values, for the tensor core
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = (1u << 4) | ((uint32_t)(PAGE >> 3) << 17) | ((uint32_t)(D >> 4) << 24);
      const uint32_t ra = smem_addr(&S.r[0][0]), va = smem_addr(&S.v[buf][0]);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = kmajor_desc(ra + part * D * D * 2 + 256 * ks);
          const uint64_t bd = kmajor_desc(va + 256 * ks);
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(idesc), "r"((part | ks) ? 1u : 0u));
        }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_addr(&S.bar_mma))
                   : "memory");
    }
    mma_pending = true;
    ok = wait_bar(&S.bar_mma, ph_mma);
    if (ok) {
      ph_mma ^= 1u;
      mma_pending = false;
    }
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
    // the next round's rotation, if it differs, while this round's codes are made
    if (r + 1 < nr && S.rmod[r + 1] != m) {
      if (tid == 0) issue_r(S.rmod[r + 1]);
      r_pending = true;
    }

    // ---- epilogue: lane o of the accumulator = output channel o ----
    float acc[PAGE];
    const uint32_t ta_addr = tmem + ((uint32_t)(32 * warp) << 16);
    tmem_ld32(ta_addr, acc);
    tmem_ld32(ta_addr + 32, acc + 32);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    const uint32_t mm0 = S.mmask[0], mm1 = S.mmask[1];
    uint32_t wr[4][4];
#pragma unroll
    for (int tau = 0; tau < 4; ++tau)
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) wr[tau][t4] = 0u;
#pragma unroll
    for (int t = 0; t < PAGE; ++t) {
      const uint32_t sel = ((t < 32 ? mm0 >> t : mm1 >> (t - 32)) & 1u);
      const uint32_t code = (uint32_t)code_of<NTHR>(acc[t] * S.sc[t], a.vthr) & (0u - sel);
      const int tt = t & 15;
      wr[t >> 4][(tt & 7) >> 1] |= code << (BITS == 2 ? 8 * (tt >> 3) + 2 * (tt & 1) : 16 * (tt >> 3) + 4 * (tt & 1));
    }
    if constexpr (BITS == 2) {
      const int sh = 16 * (iq >> 1) + 4 * (iq & 1);
#pragma unroll
      for (int tau = 0; tau < 4; ++tau)
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint32_t w = wr[tau][t4] << sh;
          w |= __shfl_xor_sync(0xffffffffu, w, 8);
          w |= __shfl_xor_sync(0xffffffffu, w, 16);
          if (t4 == iq) pw[tau][0] |= w;
        }
    } else {
      const int sh = 8 * (iq & 1);
#pragma unroll
      for (int tau = 0; tau < 4; ++tau)
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint32_t w = wr[tau][t4] << sh;
          w |= __shfl_xor_sync(0xffffffffu, w, 8);
          if ((t4 >> 1) == (iq & 1)) pw[tau][t4 & 1] |= w;
        }
    }
    // the page's last round: store its chunk words (older tokens of a tile kept)
    if (r + 1 == nr || S.rpage[r + 1] != p) {
#pragma unroll
      for (int tau = 0; tau < 4; ++tau) {
        if (TILE * tau + TILE <= ta || TILE * tau >= tb) continue;
        uint32_t *tw = reinterpret_cast<uint32_t *>(pg + PL.off_v + tau * PL.tile_bytes);
#pragma unroll
        for (int k = 0; k < PW; ++k) {
          const int t4 = BITS == 2 ? iq : 2 * (iq & 1) + k;
          uint32_t *dst = BITS == 2 ? tw + (4 * gq + t4) * 4 + warp : tw + (4 * gq + t4) * 8 + 2 * warp + (iq >> 1);
          uint32_t val = pw[tau][k];
          if (TILE * tau < ta) val |= *dst & v_keep_mask<BITS>(t4, ta - TILE * tau);
          *dst = val;
        }
      }
    }
    tc_fence_before();
    __syncthreads();                               // accumulator and per-round arrays free again
  }
  cp_async_wait<0>();
  if (failed) {
    if (tid == 0) atomicOr(a.err, ERR_WAIT);
    if (r_pending) (void)wait_bar(&S.bar_r, ph_r);
    if (mma_pending) (void)wait_bar(&S.bar_mma, ph_mma);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(V_TMEM_COLS));
}

// Shared memory of the key kernel: rotated keys, their codes and group statistics.
struct KeySmem {
  float xt[PAGE * D];              // keys [token][c] (rotated, fp32)
  uint8_t kc[PAGE * D];            // key codes of the page
  float kmn[2][D], kmx[2][D];     // group min and range (fp16 values held as fp32)
  float red[2][2][D];              // per-half min / max of a group
};

// ---------------------------------------------------------------------------
// Keys: the groups that complete with this chunk (or every new token for
// TurboQuant keys), and the new fp16 tail
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(THREADS) append_key_kernel(const AppendArgs a) {
  constexpr int NTHR = (1 << BITS) - 1;
  extern __shared__ __align__(128) unsigned char smem_raw[];
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

template <int BITS>
cudaError_t set_append_attrs() {
  cudaError_t r = cudaFuncSetAttribute(append_value_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(ValueSmem));
  if (r == cudaSuccess)
    r = cudaFuncSetAttribute(append_key_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(KeySmem));
  if (r == cudaSuccess)
    r = cudaFuncSetAttribute(append_key_kernel<BITS>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
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
    cudaError_t r = set_append_attrs<2>();
    if (r == cudaSuccess) r = set_append_attrs<4>();
    return r;
  });
  if (e != cudaSuccess) return e;
  if (a.vppc < 1 || a.vppc > V_MAX_PPC) return cudaErrorInvalidValue;
  const dim3 kgrid(n_pages, a.L * a.Hkv), vgrid((n_pages + a.vppc - 1) / a.vppc, a.L * a.Hkv);
  if ((e = cudaEventRecord(fork, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(aux, fork, 0)) != cudaSuccess) return e;
  if (a.bits == 2) append_key_kernel<2><<<kgrid, THREADS, sizeof(KeySmem), aux>>>(a);
  else append_key_kernel<4><<<kgrid, THREADS, sizeof(KeySmem), aux>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.bits == 2) append_value_kernel<2><<<vgrid, VTHREADS, sizeof(ValueSmem), s>>>(a);
  else append_value_kernel<4><<<vgrid, VTHREADS, sizeof(ValueSmem), s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaEventRecord(join, aux)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(s, join, 0);
}

}  // namespace okvq
