// Token-by-token (recurrent) forward of the gated delta rule, for decoding a
// few tokens per sequence after a chunked prefill:
//   S <- exp(g_t) S;  S <- S + beta_t (v_t - S k_t) k_t^T;  o_t = S q_t
// (the recurrence as stated on the onedev.kr summary of the FlashQLA talk,
// linear-attention background paragraph; decoding is the agentic-inference
// use named on the tilnote.io note, section on the workloads it wins).
//
// The rows of S (value features) evolve independently: row i only needs v_t[i]
// and the shared k_t, q_t.  So a warp keeps RPW rows of S in registers (lane l
// holds features [l * D/32, (l+1) * D/32)) across the token loop; the two row
// dot products per token are warp butterflies.  Grid: (sequence x head,
// D / (8 * RPW)) CTAs of 8 warps.  HBM traffic is the state read and written
// once per call plus the token inputs, all in coalesced 16-byte (or 8-byte)
// accesses.  The token inputs are staged in shared memory 16 tokens at a time
// (k normalised and q scaled once per CTA), so the token loop waits on shared
// memory, not on global loads.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int RPW = 8;  // state rows per warp (the joint reductions below assume eight)
constexpr int TB = 16;  // tokens staged in shared memory at a time

__device__ __forceinline__ float bsum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Eight per-lane values v[0..7] -> lane l gets the warp sum of v[l >> 2], i.e. row r's sum sits in
// lanes 4r .. 4r+3 (transpose-reduce: 9 shuffles instead of 8 x 5).
__device__ __forceinline__ float tsum8(const float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = (b4 ? v[4 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[4 + i], 16);
  float c[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) c[i] = (b3 ? a[2 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[2 + i], 8);
  float d = (b2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, b2 ? c[0] : c[1], 4);
  d += __shfl_xor_sync(0xffffffffu, d, 2);
  d += __shfl_xor_sync(0xffffffffu, d, 1);
  return d;
}

template <typename I, int EPL>
__device__ __forceinline__ void load_vec(const I *p, float (&x)[EPL]) {
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] = tof(p[e]);
}

template <int D>
__device__ __forceinline__ void load_row(const float *p, float (&x)[D / 32]) {
  if constexpr (D == 128) {
    const float4 t = *reinterpret_cast<const float4 *>(p);
    x[0] = t.x;
    x[1] = t.y;
    x[2] = t.z;
    x[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2 *>(p);
    x[0] = t.x;
    x[1] = t.y;
  }
}

template <int D>
__device__ __forceinline__ void store_row(float *p, const float (&x)[D / 32]) {
  if constexpr (D == 128) *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  else *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
}

}  // namespace

template <typename I, int D>
__global__ void __launch_bounds__(256) recurrent_kernel(RecArgs a) {
  constexpr int EPL = D / 32;
  const int nh = blockIdx.x, H = a.H, n = nh / H, h = nh % H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rowc = blockIdx.y * 8 * RPW;  // this CTA's first state row
  const int row0 = rowc + warp * RPW;     // this warp's
  const size_t sbase = (size_t)nh * D * D;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const I *q = static_cast<const I *>(a.q);
  const I *k = static_cast<const I *>(a.k);
  const I *v = static_cast<const I *>(a.v);
  I *o = static_cast<I *>(a.o);
  // the token inputs of TB tokens at a time, staged in shared memory with k normalised and q scaled once
  // per CTA (not once per warp), so that the token loop reads them at shared-memory latency
  __shared__ __align__(16) float ks[TB][D], qs[TB][D], vs[TB][8 * RPW];
  __shared__ float as[TB], bs[TB];

  float s[RPW][EPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    if (a.S_in) {
      load_row<D>(a.S_in + sbase + (size_t)(row0 + r) * D + lane * EPL, s[r]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) s[r][e] = 0.f;
    }
  }

  for (int t0 = 0; t0 < a.T; t0 += TB) {
    const int nt = min(TB, a.T - t0);
    // ---- stage tokens t0 .. t0 + nt - 1: warp w takes tokens w, w + 8 (k, q and their norms); every
    // thread four of the CTA's v entries; threads 0 .. nt - 1 the gates
    for (int tt = warp; tt < nt; tt += 8) {
      const size_t tok = ((size_t)n * a.T + t0 + tt) * H + h;
      float kk[EPL], qq[EPL];
      load_vec<I, EPL>(k + tok * D + lane * EPL, kk);
      load_vec<I, EPL>(q + tok * D + lane * EPL, qq);
      float km = 1.f, qm = a.scale;
      if (l2) {
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          sk = fmaf(kk[e], kk[e], sk);
          sq = fmaf(qq[e], qq[e], sq);
        }
        km = rsqrtf(bsum(sk) + 1e-6f);
        qm *= rsqrtf(bsum(sq) + 1e-6f);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        ks[tt][lane * EPL + e] = kk[e] * km;
        qs[tt][lane * EPL + e] = qq[e] * qm;
      }
    }
    for (int i = threadIdx.x; i < nt * 8 * RPW; i += blockDim.x) {
      const int tt = i / (8 * RPW), r = i % (8 * RPW);
      vs[tt][r] = tof(v[(((size_t)n * a.T + t0 + tt) * H + h) * D + rowc + r]);
    }
    if (threadIdx.x < nt) {
      const size_t tok = ((size_t)n * a.T + t0 + threadIdx.x) * H + h;
      as[threadIdx.x] = expf(a.g[tok]);
      bs[threadIdx.x] = a.beta[tok];
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      float kk[EPL], qq[EPL], vv[RPW];
      load_row<D>(&ks[tt][lane * EPL], kk);
      load_row<D>(&qs[tt][lane * EPL], qq);
#pragma unroll
      for (int r = 0; r < RPW; r += 4) {
        const float4 t4 = *reinterpret_cast<const float4 *>(&vs[tt][warp * RPW + r]);
        vv[r] = t4.x;
        vv[r + 1] = t4.y;
        vv[r + 2] = t4.z;
        vv[r + 3] = t4.w;
      }
      const float alpha = as[tt], bt = bs[tt];
      float dk[RPW], dq[RPW];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        dk[r] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          s[r][e] *= alpha;
          dk[r] = fmaf(s[r][e], kk[e], dk[r]);
        }
      }
      const float dkr = tsum8(dk);  // row (lane >> 2)'s S k, then broadcast to every lane
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const float u = bt * (vv[r] - __shfl_sync(0xffffffffu, dkr, 4 * r));
        dq[r] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          s[r][e] = fmaf(u, kk[e], s[r][e]);
          dq[r] = fmaf(s[r][e], qq[e], dq[r]);
        }
      }
      const float out = tsum8(dq);  // row (lane >> 2)'s S q
      if ((lane & 3) == 0) o[(((size_t)n * a.T + t0 + tt) * H + h) * D + row0 + (lane >> 2)] = fromf<I>(out);
    }
    __syncthreads();  // the staged block is read before the next one overwrites it
  }

#pragma unroll
  for (int r = 0; r < RPW; ++r) store_row<D>(a.S_out + sbase + (size_t)(row0 + r) * D + lane * EPL, s[r]);
}

int launch_recurrent(const RecArgs &a, bool is_bf16, int D, int NH, cudaStream_t st) {
  if (NH == 0) return 0;
  const dim3 grid(NH, D / (8 * RPW));
  if (is_bf16 && D == 128) recurrent_kernel<bf16, 128><<<grid, 256, 0, st>>>(a);
  else if (is_bf16 && D == 64) recurrent_kernel<bf16, 64><<<grid, 256, 0, st>>>(a);
  else if (!is_bf16 && D == 128) recurrent_kernel<float, 128><<<grid, 256, 0, st>>>(a);
  else if (!is_bf16 && D == 64) recurrent_kernel<float, 64><<<grid, 256, 0, st>>>(a);
  else return -1;
  return (int)cudaGetLastError();
}

}  // namespace gdn
