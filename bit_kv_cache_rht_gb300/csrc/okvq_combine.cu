// Merge of the split-K decode partials ("OmniKVQuant: KV Cache Quantization for
// Omni-LLMs", section 1 INTRODUCTION, Implementation bullet: the inverse value
// rotations are batched after attention aggregation).
//
// combine_kernel - per (unit, 32 output channels): log-sum-exp merge of the unit's
//   partials (and of the far-memory partials, if any), then
//   O = (sum_m R_m^T o_m) / (l sqrt d) on the tensor cores, plus the far-memory
//   values, fp16 store.
#include "okvq_device.h"

namespace okvq {

namespace {

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// One CTA per (unit, 64 output channels): merge the unit's partials by
// log-sum-exp (warp w = query head w), then O^T[c][h] = sum_r R^T[c][r] o[h][r] / l
// on the tensor cores. R^T comes pre-split into fp16 high and residual parts in
// mma fragment order (one bulk copy per CTA, issued before the wait on the decode
// grid); o / l is split the same way, and hi*hi + hi*lo + lo*hi carries the
// product to ~2^-22 relative (fp32 accumulation).
#ifndef OKVQ_CB_CH
#define OKVQ_CB_CH 32
#endif
constexpr int CB_CH = OKVQ_CB_CH;               // output channels per CTA (32 or 64)
constexpr int CB_MT = CB_CH / 16;               // m-tiles of 16 channels per CTA
constexpr int CB_KS = 8 / CB_MT;                // warps sharing an m-tile, each a slice of the k-steps
constexpr int CB_RED = (CB_KS - 1) * CB_MT * 32 * 4;   // floats of the cross-warp k-slice reduction
constexpr int OSTRIDE = MAXM * D + 4;           // padded row of the merged o (floats)
__global__ void __launch_bounds__(256, 1) combine_kernel(const CombineArgs a) {
  extern __shared__ __align__(128) unsigned char csm[];
  uint4 *afr = reinterpret_cast<uint4 *>(csm);                                  // [MT][8M][32][2] hi|lo
  float *osh = reinterpret_cast<float *>(csm + CB_MT * 8 * MAXM * 32 * 32);       // [8][OSTRIDE]
  float *red = osh + MAXGQ * OSTRIDE;                                             // [KS-1][MT][32][4]
  float *ofar = red + CB_RED;                                                      // [8][CB_CH] far memory / l
  __shared__ __align__(8) uint64_t bar;
  const int unit = blockIdx.x, half = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, t4 = lane & 3;
  const int gq = a.Hq / a.Hkv;
  const int s0 = a.unit_seg[unit], s1 = a.unit_seg[unit + 1];
  const int lh = unit % (a.L * a.Hkv);
  const int nks = 8 * a.M;                                // 16-row k-steps over the stacked R_m
  const uint32_t fbytes = (uint32_t)(CB_MT * nks * 32 * 32);
  if (tid == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
    bulk_load(afr, a.rot_frag + ((long long)lh * 8 + CB_MT * half) * nks * 32 * 2, fbytes, &bar);
  }
  // everything above only reads the rotations; the partials come from the decode grid.
  // The next decode step may launch as this grid's CTAs retire (it waits for this grid
  // before it reads or writes anything this one touches).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nr = a.M * D;
  if (w < gq) {
    constexpr int OPER = MAXM * D / 32;
    float o[OPER];
#pragma unroll
    for (int k = 0; k < OPER; ++k) o[k] = 0.f;
    float L = 0.f;
    const float *pbase = a.partials + (long long)w * PARTIAL_FLOATS;
    auto part = [&](int s) { return pbase + (long long)s * MAXGQ * PARTIAL_FLOATS; };
    // the first two segments' o rows are loaded with the (m, l) pairs: one round
    // trip to L2 fewer for the common unit of one or two segments
    float p0[OPER], p1[OPER];
#pragma unroll
    for (int k = 0; k < OPER; ++k) {
      // lane: channels 2 lane + 64 (k / 2) + (k % 2), as 8-byte pairs
      p0[k] = (s0 < s1 && 64 * (k >> 1) < nr) ? part(s0)[2 + 2 * lane + 64 * (k >> 1) + (k & 1)] : 0.f;
      p1[k] = (s0 + 1 < s1 && 64 * (k >> 1) < nr) ? part(s0 + 1)[2 + 2 * lane + 64 * (k >> 1) + (k & 1)] : 0.f;
    }
    float m0 = -INFINITY, l0 = 0.f;
    if (s0 + lane < s1) {
      const float2 ml = *reinterpret_cast<const float2 *>(part(s0 + lane));
      m0 = ml.x;
      l0 = ml.y;
    }
    float M = m0;
    for (int s = s0 + 32 + lane; s < s1; s += 32) M = fmaxf(M, part(s)[0]);
    // far-memory partials of this unit and head: m, l, o[D] in the original value basis
    const float *fbase = a.far_split ? a.far + ((long long)unit * a.far_split * MAXGQ + w) * FAR_PARTIAL_FLOATS : a.far;
    auto farp = [&](int f) { return fbase + (long long)f * MAXGQ * FAR_PARTIAL_FLOATS; };
    for (int f = lane; f < a.far_split; f += 32) M = fmaxf(M, farp(f)[0]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float of[CB_CH / 32] = {};             // channels half * CB_CH + lane (+ 32)
    for (int f = 0; f < a.far_split; ++f) {
      const float mf = farp(f)[0];
      const float wt = mf == -INFINITY ? 0.f : ex2(mf - M);
      if (lane == 0) L = fmaf(wt, farp(f)[1], L);
#pragma unroll
      for (int j = 0; j < CB_CH / 32; ++j) of[j] = fmaf(wt, farp(f)[2 + half * CB_CH + lane + 32 * j], of[j]);
    }
    for (int sb = s0; sb < s1; sb += 32) {
      float wt = 0.f;
      if (sb + lane < s1) {
        float m = m0, l = l0;
        if (sb != s0) {
          const float2 ml = *reinterpret_cast<const float2 *>(part(sb + lane));
          m = ml.x;
          l = ml.y;
        }
        wt = m == -INFINITY ? 0.f : ex2(m - M);
        L = fmaf(wt, l, L);
      }
      const int n = min(32, s1 - sb);
      int j0 = 0;
      if (sb == s0) {                     // lane 1's weight is 0 (and p1 = 0) without a second segment
        const float w0 = __shfl_sync(0xffffffffu, wt, 0), w1 = __shfl_sync(0xffffffffu, wt, 1);
#pragma unroll
        for (int k = 0; k < OPER; ++k) {
          o[k] = fmaf(w0, p0[k], o[k]);
          o[k] = fmaf(w1, p1[k], o[k]);
        }
        j0 = 2;
      }
#pragma unroll 4
      for (int j = j0; j < n; ++j) {
        const float ws = __shfl_sync(0xffffffffu, wt, j);
        const float *p = part(sb + j) + 2 + lane;
#pragma unroll
        for (int k = 0; k < OPER; k += 2)
          if (64 * (k >> 1) < nr) {
            const float2 v = *reinterpret_cast<const float2 *>(p + lane + 64 * (k >> 1));
            o[k] = fmaf(ws, v.x, o[k]);
            o[k + 1] = fmaf(ws, v.y, o[k + 1]);
          }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int k = 0; k < OPER; k += 2)
      if (64 * (k >> 1) < nr)
        *reinterpret_cast<float2 *>(osh + w * OSTRIDE + 2 * lane + 64 * (k >> 1)) = make_float2(o[k] * inv, o[k + 1] * inv);
#pragma unroll
    for (int j = 0; j < CB_CH / 32; ++j) ofar[w * CB_CH + lane + 32 * j] = of[j] * inv;
  } else if (w < MAXGQ) {
    for (int k = lane; k < nr; k += 32) osh[w * OSTRIDE + k] = 0.f;
#pragma unroll
    for (int j = 0; j < CB_CH / 32; ++j) ofar[w * CB_CH + lane + 32 * j] = 0.f;
  }
  __syncthreads();
  const bool got = mbar_wait(&bar, 0);
  if (!got && tid == 0) atomicOr(a.err, ERR_WAIT);
  // warp w: m-tile w % MT of this CTA's channels, k-step slice w / MT
  const int mtl = w % CB_MT, kh = w / CB_MT, k0 = kh * (nks / CB_KS), k1 = k0 + nks / CB_KS;
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  if (got) {
    for (int ks = k0; ks < k1; ++ks) {
      const uint4 ah = afr[((mtl * nks + ks) * 32 + lane) * 2];
      const uint4 al = afr[((mtl * nks + ks) * 32 + lane) * 2 + 1];
      const uint32_t Ah[4] = {ah.x, ah.y, ah.z, ah.w}, Al[4] = {al.x, al.y, al.z, al.w};
      const float2 x01 = *reinterpret_cast<const float2 *>(osh + g * OSTRIDE + 16 * ks + 2 * t4);
      const float2 x89 = *reinterpret_cast<const float2 *>(osh + g * OSTRIDE + 16 * ks + 2 * t4 + 8);
      const __half2 h01 = __floats2half2_rn(x01.x, x01.y), h89 = __floats2half2_rn(x89.x, x89.y);
      const float2 f01 = __half22float2(h01), f89 = __half22float2(h89);
      const uint32_t bh0 = h2u(h01), bh1 = h2u(h89);
      const uint32_t bl0 = pack_h2(x01.x - f01.x, x01.y - f01.y), bl1 = pack_h2(x89.x - f89.x, x89.y - f89.y);
      mma16816(d, Ah, bh0, bh1);
      mma16816(d, Ah, bl0, bl1);
      mma16816(d, Al, bh0, bh1);
    }
  }
  if (kh > 0)
    *reinterpret_cast<float4 *>(red + (((kh - 1) * CB_MT + mtl) * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
  __syncthreads();
  if (kh == 0 && got) {
    float y[4] = {d[0], d[1], d[2], d[3]};
#pragma unroll
    for (int k = 1; k < CB_KS; ++k) {
      const float4 e = *reinterpret_cast<const float4 *>(red + (((k - 1) * CB_MT + mtl) * 32 + lane) * 4);
      y[0] += e.x; y[1] += e.y; y[2] += e.z; y[3] += e.w;
    }
    const int session = unit / (a.L * a.Hkv);
    const int layer = lh / a.Hkv, kvh = lh % a.Hkv;
    __half *ob = a.out + (((long long)session * a.L + layer) * a.Hq + kvh * gq) * D;
    const int c = half * CB_CH + 16 * mtl + g;
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const int h = 2 * t4 + (e2 & 1), cc = c + 8 * (e2 >> 1);
      if (h < gq) ob[h * D + cc] = __float2half_rn(fmaf(y[e2], INV_SQRT_D, ofar[h * CB_CH + cc - half * CB_CH]));
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
  if (a.units <= 0) return cudaSuccess;
  static std::atomic<uint64_t> attr_done{0};
  const size_t smem = (size_t)CB_MT * 8 * MAXM * 32 * 32 + (MAXGQ * OSTRIDE + CB_RED + MAXGQ * CB_CH) * sizeof(float);
  cudaError_t ea = once_per_device(attr_done, [&] {
    cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // same shared/L1 split as the decode kernel: no reconfiguration between the two
    return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  });
  if (ea != cudaSuccess) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.units, D / CB_CH);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace okvq
