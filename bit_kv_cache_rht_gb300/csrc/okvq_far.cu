// Far-memory pseudo tokens ("ProtoKV: Streaming Video Understanding under
// Delayed Query with Summary-State Memory", section 3.3 Eq. (2), Appendix A.3
// Eq. (4) and Algorithm 4): pseudo tokens k~, v~ synthesized by the caller join
// the near window's softmax, each with the additive log-mass bias log n_k of its
// prototype k (inactive prototypes, n_k = 0, are skipped).
//
// far_kernel - one CTA (12 warps) per (unit, split) of the unit's pseudo tokens.
//   Each warp streams 16-token stages of fp16 keys and values through a private
//   2-stage shared ring (one bulk copy per 256-byte row into rows padded to 272
//   bytes, so that the ldmatrix row reads below hit distinct banks; mbarrier
//   completion, bounded waits) and computes, per 16-token m-tile,
//     scores  S[16 tok x 8 heads] = K~[16 x 128] * q^T[128 x 8]     (8 MMAs)
//     softmax online, base 2, per head column, lazy reference
//     values  O^T[128 ch x 8 heads] += V~^T[128 x 16] * P[16 x 8]   (8 MMAs)
//   (P moves from the score fragment layout to the value B fragment with two
//   8x8 register transposes). Warps merge in shared memory; one partial
//   (m, l, o[128]) per (split, head) goes to the merge kernel, which adds it to
//   the near window's partials in the original value basis.
#include "okvq_device.h"

namespace okvq {

namespace {

#ifndef OKVQ_FAR_WARPS
#define OKVQ_FAR_WARPS 12
#endif
#ifndef OKVQ_FAR_TOK
#define OKVQ_FAR_TOK 16
#endif
#ifndef OKVQ_FAR_STAGES
#define OKVQ_FAR_STAGES 2
#endif
constexpr int FAR_WARPS = OKVQ_FAR_WARPS;
constexpr int FAR_TOK = OKVQ_FAR_TOK;       // tokens per stage (16 or 32)
constexpr int FAR_STAGES = OKVQ_FAR_STAGES;
constexpr int FAR_MT = FAR_TOK / 16;        // 16-token m-tiles per stage
static_assert(FAR_TOK == 16 || FAR_TOK == 32, "stage of one or two m-tiles");
constexpr int FAR_ROW = D * 2 + 16;         // padded row (bytes)
constexpr int FAR_STAGE_BYTES = 2 * FAR_TOK * FAR_ROW;   // K rows then V rows
constexpr float HEADROOM = 6.0f;            // log2 units, as in the near kernel

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ void bulk_row(uint32_t dst, const void *src, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "n"(D * 2), "r"(smem_u32(bar))
      : "memory");
}

struct FarMerge {
  float m[FAR_WARPS][MAXGQ];
  float l[FAR_WARPS][MAXGQ];
  float o[FAR_WARPS][MAXGQ][D + 4];
};

__global__ void __launch_bounds__(FAR_WARPS * 32, 1) far_kernel(const FarArgs a) {
  extern __shared__ __align__(128) unsigned char fsm[];
  __shared__ __align__(8) uint64_t bars[FAR_WARPS][FAR_STAGES];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
  const long long item = blockIdx.x;
  const long long unit = item / a.nsplit;
  const int split = (int)(item % a.nsplit);
  const int lh = (int)(unit % (a.L * a.Hkv)), session = (int)(unit / (a.L * a.Hkv));
  const int layer = lh / a.Hkv, kvh = lh % a.Hkv;
  const int gq = a.Hq / a.Hkv;
  const int t0 = split * a.chunk, t1 = min(a.n_far, t0 + a.chunk);
  const int nstage = t1 > t0 ? (t1 - t0 + FAR_TOK - 1) / FAR_TOK : 0;
  const int my_n = nstage > warp ? (nstage - warp + FAR_WARPS - 1) / FAR_WARPS : 0;
  unsigned char *ring = fsm + (size_t)warp * FAR_STAGES * FAR_STAGE_BYTES;
  const __half *kbase = a.k + (long long)unit * a.n_far * D;
  const __half *vbase = a.v + (long long)unit * a.n_far * D;
  const float *mass = a.mass + (long long)unit * (a.n_far / a.per_proto);

  if (lane == 0)
    for (int s = 0; s < FAR_STAGES; ++s) mbar_init(&bars[warp][s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  // the merge kernel may be scheduled as SMs free up; it waits for this grid's memory
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // issue stage k of this warp (tokens t0 + 32 (warp + 4k) ...): one arrival with the
  // byte count, then each lane copies its own K and V rows
  auto issue = [&](int k) {
    const int st = k % FAR_STAGES;
    const int s0 = t0 + FAR_TOK * (warp + FAR_WARPS * k);
    const int nt = min(FAR_TOK, t1 - s0);
    if (lane == 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bars[warp][st])),
                   "r"((uint32_t)(2 * nt * D * 2))
                   : "memory");
    }
    __syncwarp();                                  // the stage's earlier reads are done
    fence_async_smem();
    unsigned char *stp = ring + (size_t)st * FAR_STAGE_BYTES;
    if (lane < nt) {
      const uint32_t dst = smem_u32(stp);
      bulk_row(dst + lane * FAR_ROW, kbase + (long long)(s0 + lane) * D, &bars[warp][st]);
      bulk_row(dst + (FAR_TOK + lane) * FAR_ROW, vbase + (long long)(s0 + lane) * D, &bars[warp][st]);
    } else if (lane < FAR_TOK) {
      // rows past the last token: zeros, so that their (zero-weighted) values stay finite
      uint4 *kr = reinterpret_cast<uint4 *>(stp + lane * FAR_ROW);
      uint4 *vr = reinterpret_cast<uint4 *>(stp + (FAR_TOK + lane) * FAR_ROW);
#pragma unroll
      for (int i = 0; i < D * 2 / 16; ++i) kr[i] = vr[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  for (int k = 0; k < min(my_n, FAR_STAGES); ++k) issue(k);

  // query B fragments (channels x heads): head g, channels 16kb + 2t4 (+1), (+8, +9)
  uint32_t qb[8][2];
  {
    const __half *qs = a.q + (((long long)session * a.L + layer) * a.Hq + (long long)kvh * gq) * D;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      qb[kb][0] = g < gq ? *reinterpret_cast<const uint32_t *>(qs + g * D + 16 * kb + 2 * t4) : 0u;
      qb[kb][1] = g < gq ? *reinterpret_cast<const uint32_t *>(qs + g * D + 16 * kb + 2 * t4 + 8) : 0u;
    }
  }

  float acc[8][4];            // O^T: channel 16mt + g (+8) x heads 2t4, 2t4+1
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};   // heads 2t4, 2t4+1
  bool wait_failed = false;
  int k_stop = my_n;
  // ldmatrix lane roles: row (lane & 7) + 8 ((lane >> 3) & 1), 16-byte column (lane >> 4)
  const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lcol = 16 * (lane >> 4);
  // the transposed load for V: token (lane & 7) + 8 (lane >> 4), channel column 8 ((lane >> 3) & 1)
  const int vrow = (lane & 7) + 8 * (lane >> 4), vcol = 16 * ((lane >> 3) & 1);

  for (int k = 0; k < my_n; ++k) {
    const int st = k % FAR_STAGES;
    if (!mbar_wait(&bars[warp][st], (uint32_t)((k / FAR_STAGES) & 1))) {
      wait_failed = true;
      k_stop = k;
      break;
    }
    const int s0 = t0 + FAR_TOK * (warp + FAR_WARPS * k);
    const uint32_t kst = smem_u32(ring + (size_t)st * FAR_STAGE_BYTES);
    const uint32_t vst = kst + FAR_TOK * FAR_ROW;
    // ---- scores of the stage's 16-token m-tiles ----
    float sc[FAR_MT][4];
#pragma unroll
    for (int mtile = 0; mtile < FAR_MT; ++mtile) {
      float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        uint32_t A[4];
        ldsm_x4(kst + (16 * mtile + lrow) * FAR_ROW + 32 * kb + lcol, A);
        mma16816(d4, A, qb[kb][0], qb[kb][1]);
      }
      // rows = tokens g, g + 8 of the m-tile; columns = heads 2t4, 2t4 + 1
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = s0 + 16 * mtile + g + 8 * r;
        const float n = tok < t1 ? mass[tok / a.per_proto] : 0.f;
        const bool on = n > 0.f;                 // inactive prototype or past the end: no weight
        const float bias = on ? log2f(n) : 0.f;
        sc[mtile][2 * r] = on ? fmaf(d4[2 * r], INV_SQRT_D * LOG2E, bias) : -INFINITY;
        sc[mtile][2 * r + 1] = on ? fmaf(d4[2 * r + 1], INV_SQRT_D * LOG2E, bias) : -INFINITY;
      }
    }
    // ---- online softmax per head column (lanes with the same t4 hold the same heads) ----
    float mx[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[e] = fmaxf(sc[0][e], sc[0][2 + e]);
#pragma unroll
      for (int mtile = 1; mtile < FAR_MT; ++mtile) mx[e] = fmaxf(mx[e], fmaxf(sc[mtile][e], sc[mtile][2 + e]));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(FULL, mx[e], 4));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(FULL, mx[e], 8));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(FULL, mx[e], 16));
    }
    const bool up0 = mx[0] > m_run[0], up1 = mx[1] > m_run[1];
    if (__any_sync(FULL, up0 || up1)) {
      const float n0 = up0 ? mx[0] + HEADROOM : m_run[0], n1 = up1 ? mx[1] + HEADROOM : m_run[1];
      const float f0 = m_run[0] == -INFINITY ? 0.f : ex2(m_run[0] - n0);
      const float f1 = m_run[1] == -INFINITY ? 0.f : ex2(m_run[1] - n1);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[mt][0] *= f0; acc[mt][2] *= f0;
        acc[mt][1] *= f1; acc[mt][3] *= f1;
      }
      l_run[0] *= f0;
      l_run[1] *= f1;
      m_run[0] = n0;
      m_run[1] = n1;
    }
    uint32_t pb[FAR_MT][2];   // value B fragments per m-tile: tokens 0-7 | 8-15
#pragma unroll
    for (int mtile = 0; mtile < FAR_MT; ++mtile) {
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        p[i] = m_run[i & 1] == -INFINITY ? 0.f : ex2(sc[mtile][i] - m_run[i & 1]);
        l_run[i & 1] += p[i];
      }
      pb[mtile][0] = movm_t(pack2(p[0], p[1]));
      pb[mtile][1] = movm_t(pack2(p[2], p[3]));
    }
    // ---- values ----
#pragma unroll
    for (int mtile = 0; mtile < FAR_MT; ++mtile) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t A[4];
        ldsm_x4_t(vst + (16 * mtile + vrow) * FAR_ROW + 32 * mt + vcol, A);
        mma16816(acc[mt], A, pb[mtile][0], pb[mtile][1]);
      }
    }
    __syncwarp();
    if (k + FAR_STAGES < my_n) issue(k + FAR_STAGES);
  }
  if (__syncthreads_or(wait_failed)) {
    if (tid == 0) atomicOr(a.err, ERR_WAIT);
    // give copies still in flight a bounded chance to land before the CTA exits
    if (lane == 0)
      for (int k = k_stop; k < min(my_n, k_stop + FAR_STAGES); ++k)
        (void)mbar_wait(&bars[warp][k % FAR_STAGES], (uint32_t)((k / FAR_STAGES) & 1));
    return;
  }

  // ---- warp totals, then merge the 4 warps (the rings are free now) ----
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    l_run[e] += __shfl_xor_sync(FULL, l_run[e], 4);
    l_run[e] += __shfl_xor_sync(FULL, l_run[e], 8);
    l_run[e] += __shfl_xor_sync(FULL, l_run[e], 16);
  }
  FarMerge &MG = *reinterpret_cast<FarMerge *>(fsm);
  if (g == 0) {
    MG.m[warp][2 * t4] = m_run[0];
    MG.m[warp][2 * t4 + 1] = m_run[1];
    MG.l[warp][2 * t4] = l_run[0];
    MG.l[warp][2 * t4 + 1] = l_run[1];
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    MG.o[warp][2 * t4][16 * mt + g] = acc[mt][0];
    MG.o[warp][2 * t4 + 1][16 * mt + g] = acc[mt][1];
    MG.o[warp][2 * t4][16 * mt + g + 8] = acc[mt][2];
    MG.o[warp][2 * t4 + 1][16 * mt + g + 8] = acc[mt][3];
  }
  __syncthreads();
  float *part = a.partials + item * MAXGQ * FAR_PARTIAL_FLOATS;
  for (int i = tid; i < MAXGQ * D; i += FAR_WARPS * 32) {
    const int hh = i / D, ch = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < FAR_WARPS; ++w) M = fmaxf(M, MG.m[w][hh]);
    float o = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < FAR_WARPS; ++w) {
      const float s = MG.m[w][hh] == -INFINITY ? 0.f : ex2(MG.m[w][hh] - M);
      o = fmaf(s, MG.o[w][hh][ch], o);
      L = fmaf(s, MG.l[w][hh], L);
    }
    float *ph = part + hh * FAR_PARTIAL_FLOATS;
    if (ch == 0) {
      ph[0] = M;
      ph[1] = L;
    }
    ph[2 + ch] = o;
  }
}

}  // namespace

int far_pass_tokens() { return FAR_WARPS * FAR_TOK; }

size_t far_smem_bytes() {
  const size_t ring = (size_t)FAR_WARPS * FAR_STAGES * FAR_STAGE_BYTES;
  return ring > sizeof(FarMerge) ? ring : sizeof(FarMerge);
}

cudaError_t launch_far(const FarArgs &a, cudaStream_t s) {
  const long long items = a.units * a.nsplit;
  if (items <= 0) return cudaSuccess;
  static std::atomic<uint64_t> attr_done{0};
  const size_t smem = far_smem_bytes();
  cudaError_t e = once_per_device(attr_done, [&] {
    return cudaFuncSetAttribute(far_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  far_kernel<<<(unsigned)items, FAR_WARPS * 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace okvq
