// Value-rotation calibration ("OmniKVQuant: KV Cache Quantization for
// Omni-LLMs", section 2 METHOD, second OmniKVQuant bullet: directions are
// weighted by their contribution to attention outputs, a covariance matrix is
// computed per modality, and its eigenbasis is the modality's value rotation).
//
// calib_kernel - one CTA per ((layer, kv head), modality). The 128 x 128
//   weighted covariance is accumulated in shared memory (weighted mean first,
//   then the centered sum, one calibration token at a time), then diagonalized
//   in place by the cyclic Jacobi method in fp32: each round applies 64 disjoint
//   plane rotations (round-robin pairing, 127 rounds per sweep), rows first, then
//   columns and the eigenvector matrix, each update written as a correction of
//   the old entry (x_p - s (x_q + tau x_p), tau = s / (1 + c)), and the pair's
//   2 x 2 block set to its exact diagonal form. A pair is left alone when its off-diagonal
//   entry is negligible (below 1e-7 of the geometric mean of its two diagonal
//   entries, or below 1e-9 of the Frobenius norm); the iteration stops after a
//   sweep that rotated nothing (at most 30 sweeps). Eigenpairs are then ranked by
//   descending eigenvalue and each eigenvector signed so that its largest-magnitude
//   entry (the first one on a tie) is positive; the rotation's rows are the
//   eigenvectors.
#include "okvq_internal.h"

namespace okvq {

namespace {

constexpr int CT = 512;              // threads per CTA
constexpr int NPAIR = D / 2;         // disjoint rotations per round
constexpr int MAX_SWEEPS = 30;
constexpr float TOL_REL = 1e-7f;      // |a_pq| <= TOL_REL * sqrt(|a_pp a_qq|): converged pair
constexpr float TOL_ABS = 1e-9f;      // |a_pq| <= TOL_ABS * ||A||_F: converged pair
constexpr int LD = D + 1;            // padded row stride: a column walk across lanes hits distinct banks

struct CalibArgs {
  const __half *v;                   // [n][LH][D]
  const uint8_t *mod;                // [n]
  const float *weight;               // [n][LH] or null (all 1)
  float *rot;                        // [LH][M][D][D]
  float *eig;                        // [LH][M][D] or null
  int32_t *sweeps;                   // [LH][M] or null: sweeps run, negated when not converged
  int n, LH, M;
};

// round r of the circle schedule: pair k is (127, r) for k = 0, else ((r + k) % 127, (r - k) % 127)
__device__ __forceinline__ void round_pair(int r, int k, int &p, int &q) {
  if (k == 0) {
    p = r;
    q = D - 1;
  } else {
    p = (r + k) % (D - 1);
    q = (r - k + (D - 1)) % (D - 1);
  }
  if (p > q) {
    const int t = p;
    p = q;
    q = t;
  }
}

__global__ void __launch_bounds__(CT, 1) calib_kernel(const CalibArgs a) {
  extern __shared__ __align__(16) float sm[];
  float *A = sm;                     // [D][LD] covariance, then its rotated form
  float *V = A + D * LD;             // [D][LD] accumulated rotations (columns = eigenvectors)
  float *xs = V;                     // [D] token staging before V is used
  __shared__ float sn[NPAIR], ta[NPAIR], dp[NPAIR], dq[NPAIR];
  __shared__ int pp[NPAIR], qq[NPAIR];
  __shared__ float red[CT / 32];
  __shared__ unsigned ballot[NPAIR / 32];
  __shared__ float mu[D];
  __shared__ int rank[D];
  const int unit = blockIdx.x, m = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ri = tid >> 2, cj = (tid & 3) * 32;      // this thread's 32 entries of row ri

  // ---- weighted mean and total weight of this modality's tokens ----
  float msum = 0.f, W = 0.f;
  for (int k = 0; k < a.n; ++k) {
    if (a.mod[k] != m) continue;                       // uniform across the CTA
    const float w = a.weight ? a.weight[(long long)k * a.LH + unit] : 1.f;
    W += w;
    if (tid < D) msum = fmaf(w, __half2float(a.v[((long long)k * a.LH + unit) * D + tid]), msum);
  }
  int cnt = 0;
  for (int k = 0; k < a.n; ++k) cnt += a.mod[k] == m;
  if (tid < D) mu[tid] = W > 0.f ? msum / W : 0.f;
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.f;
  __syncthreads();
  // ---- centered weighted sum of outer products, one token at a time ----
  for (int k = 0; k < a.n; ++k) {
    if (a.mod[k] != m) continue;
    if (tid < D) xs[tid] = __half2float(a.v[((long long)k * a.LH + unit) * D + tid]) - mu[tid];
    __syncthreads();
    const float w = a.weight ? a.weight[(long long)k * a.LH + unit] : 1.f;
    const float xi = w * xs[ri];
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const float4 xj = *reinterpret_cast<const float4 *>(xs + cj + j);
      acc[j] = fmaf(xi, xj.x, acc[j]);
      acc[j + 1] = fmaf(xi, xj.y, acc[j + 1]);
      acc[j + 2] = fmaf(xi, xj.z, acc[j + 2]);
      acc[j + 3] = fmaf(xi, xj.w, acc[j + 3]);
    }
    __syncthreads();
  }
  const bool degenerate = cnt < 2 || !(W > 0.f);
  const float invW = degenerate ? 0.f : 1.f / W;
#pragma unroll
  for (int j = 0; j < 32; ++j) A[ri * LD + cj + j] = acc[j] * invW;
  for (int i = tid; i < D * D; i += CT) V[(i / D) * LD + i % D] = (i / D == i % D) ? 1.f : 0.f;
  __syncthreads();

  // ---- cyclic Jacobi ----
  float fro = 0.f;                                     // ||A||_F, unchanged by the rotations
  if (!degenerate) {
    float tot = 0.f;
    for (int i = tid; i < D * D; i += CT) {
      const float x = A[(i / D) * LD + i % D];
      tot = fmaf(x, x, tot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) red[warp] = tot;
    __syncthreads();
    for (int w = 0; w < CT / 32; ++w) fro += red[w];
    fro = sqrtf(fro);
  }
  int sweeps_run = 0;
  bool converged = true;
  for (int sweep = 0; sweep < MAX_SWEEPS && !degenerate; ++sweep) {
    bool rotated = false;
    ++sweeps_run;                              // uniform: every thread reads the same ballots
    for (int r = 0; r < D - 1; ++r) {
      if (tid < NPAIR) {
        int p, q;
        round_pair(r, tid, p, q);
        const float apq = A[p * LD + q], app = A[p * LD + p], aqq = A[q * LD + q];
        float s = 0.f, tau = 0.f, t = 0.f;
        const bool rot = fabsf(apq) > TOL_REL * sqrtf(fabsf(app * aqq)) && fabsf(apq) > TOL_ABS * fro;
        if (rot) {
          const float th = (aqq - app) / (2.f * apq);
          t = (th >= 0.f ? 1.f : -1.f) / (fabsf(th) + sqrtf(fmaf(th, th, 1.f)));
          const float c = 1.f / sqrtf(fmaf(t, t, 1.f));
          s = t * c;
          tau = s / (1.f + c);
        }
        sn[tid] = s;
        ta[tid] = tau;
        pp[tid] = p;
        qq[tid] = q;
        dp[tid] = app - t * apq;                       // the rotated 2 x 2 block, exactly diagonal
        dq[tid] = aqq + t * apq;
        const unsigned bal = __ballot_sync(0xffffffffu, rot);
        if (lane == 0) ballot[warp] = bal;
      }
      __syncthreads();
      const bool any = (ballot[0] | ballot[1]) != 0u;
      rotated |= any;
      if (!any) {
        __syncthreads();                               // ballot/cs are rewritten by the next round
        continue;
      }
      // rows p, q of A: A <- J^T A, as x_p - s (x_q + tau x_p), x_q + s (x_p - tau x_q)
      for (int e = tid; e < NPAIR * D; e += CT) {
        const int k = e / D, j = e % D;
        const int p = pp[k], q = qq[k];
        const float s = sn[k], tau = ta[k];
        const float ap = A[p * LD + j], aq = A[q * LD + j];
        A[p * LD + j] = ap - s * fmaf(tau, ap, aq);
        A[q * LD + j] = aq + s * fmaf(-tau, aq, ap);
      }
      __syncthreads();
      // columns p, q of A and V: A <- A J, V <- V J; the (p, q) block takes its exact values
      for (int e = tid; e < NPAIR * D; e += CT) {
        const int k = e / D, i = e % D;
        const int p = pp[k], q = qq[k];
        const float s = sn[k], tau = ta[k];
        const float ap = A[i * LD + p], aq = A[i * LD + q];
        float np_ = ap - s * fmaf(tau, ap, aq), nq_ = aq + s * fmaf(-tau, aq, ap);
        if (i == p) {
          np_ = dp[k];
          nq_ = 0.f;
        } else if (i == q) {
          np_ = 0.f;
          nq_ = dq[k];
        }
        A[i * LD + p] = np_;
        A[i * LD + q] = nq_;
        const float vp = V[i * LD + p], vq = V[i * LD + q];
        V[i * LD + p] = vp - s * fmaf(tau, vp, vq);
        V[i * LD + q] = vq + s * fmaf(-tau, vq, vp);
      }
      __syncthreads();
    }
    if (!rotated) break;
    if (sweep == MAX_SWEEPS - 1) converged = false;
  }
  if (a.sweeps && tid == 0) a.sweeps[unit * a.M + m] = converged ? sweeps_run : -sweeps_run;

  // ---- order by descending eigenvalue, sign, write rows ----
  if (tid < D) {
    const float li = degenerate ? 0.f : A[tid * LD + tid];
    int rk = 0;
    for (int j = 0; j < D; ++j) {
      const float lj = degenerate ? 0.f : A[j * LD + j];
      rk += (lj > li) || (lj == li && j < tid);
    }
    rank[tid] = rk;
    if (a.eig) a.eig[((long long)unit * a.M + m) * D + rk] = li;
  }
  __syncthreads();
  float *out = a.rot + ((long long)unit * a.M + m) * D * D;
  // column c of V is the eigenvector of eigenvalue A[c][c]; it becomes row rank[c]
  for (int col = warp; col < D; col += CT / 32) {
    float best = 0.f;
    int bi = D;
    for (int i = lane; i < D; i += 32) {
      const float x = V[i * LD + col];
      if (fabsf(x) > fabsf(best)) {
        best = x;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, best, o);
      const int yi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (fabsf(y) > fabsf(best) || (fabsf(y) == fabsf(best) && yi < bi)) {
        best = y;
        bi = yi;
      }
    }
    const float sgn = best < 0.f ? -1.f : 1.f;
    float *row = out + (long long)rank[col] * D;
    for (int i = lane; i < D; i += 32) row[i] = sgn * V[i * LD + col];
  }
}

}  // namespace

}  // namespace okvq

using namespace okvq;

extern "C" okvq_status okvq_calibrate_rotations(int32_t num_layers, int32_t num_kv_heads, int32_t num_modalities,
                                                 const void *v, const uint8_t *modality, const float *weight,
                                                 int32_t num_tokens, float *rot_out, float *eig_out,
                                                 int32_t *sweeps_out, void *stream) {
  if (num_layers < 1 || num_kv_heads < 1 || num_modalities < 1 || num_modalities > MAXM || num_tokens < 0)
    return OKVQ_EINVAL;
  if (!is_device_memory(rot_out) || (eig_out && !is_device_memory(eig_out)) ||
      (sweeps_out && !is_device_memory(sweeps_out)))
    return OKVQ_EINVAL;
  if (num_tokens > 0 && (!is_device_memory(v) || !is_device_memory(modality) || (weight && !is_device_memory(weight))))
    return OKVQ_EINVAL;
  CalibArgs a;
  a.v = static_cast<const __half *>(v);
  a.mod = modality;
  a.weight = weight;
  a.rot = rot_out;
  a.eig = eig_out;
  a.sweeps = sweeps_out;
  a.n = num_tokens;
  a.LH = num_layers * num_kv_heads;
  a.M = num_modalities;
  const size_t smem = 2 * (size_t)D * LD * sizeof(float);
  static std::atomic<uint64_t> attr_done{0};
  if (once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(calib_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      }) != cudaSuccess)
    return OKVQ_ECUDA;
  calib_kernel<<<dim3((unsigned)a.LH, (unsigned)a.M), CT, smem, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? OKVQ_OK : OKVQ_ECUDA;
}
