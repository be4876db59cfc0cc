// Token-by-token (recurrent) forward of the gated delta rule, for decoding a
// few tokens per sequence after a chunked prefill:
//   S <- exp(g_t) S;  S <- S + beta_t (v_t - S k_t) k_t^T;  o_t = S q_t
// (the recurrence as stated on the onedev.kr summary of the FlashQLA talk,
// linear-attention background paragraph; decoding is the agentic-inference
// use named on the tilnote.io note, section on the workloads it wins).
//
// The rows of S (value features) evolve independently: row i only needs v_t[i]
// and the shared k_t, q_t.  With u = beta_t (v_t - alpha_t S_{t-1} k_t) the step
// is S_t = alpha_t S_{t-1} + u k_t^T and o_t = alpha_t S_{t-1} q_t + u (k_t . q_t),
// so both row dot products of a token read the state before the update and are
// reduced together; the update waits only for u.  A warp keeps 8 rows of S in
// registers across the token loop: a group of D/8 lanes holds R = D/32 rows
// (4 at d = 128, 2 at d = 64), each lane 8 features of each row as two float4
// pieces (piece m of lane j holds features 4 (m D/8 + j) .. + 3, so that a
// warp's 16-byte shared-memory reads of k or q hit distinct banks).  Products
// and updates are packed two-wide fp32 FMAs; the 2R dot-product parts of a lane
// are reduced over its group in one transposed butterfly.  Grid: (sequence x
// head, D / 64) CTAs of 8 warps.  HBM traffic is the state read and written
// once per call plus the token inputs, in coalesced 16-byte accesses.  The
// token inputs are staged in shared memory 16 tokens at a time (k normalised, q
// scaled and k . q formed once per CTA), so the token loop waits on shared
// memory, not on global loads.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int FPL = 8;    // features per lane of each of its rows
constexpr int WARPS = 8;  // warps per CTA, 8 state rows each
constexpr int RPC = 8 * WARPS;  // state rows per CTA
constexpr int TB = 16;    // tokens staged in shared memory at a time

__device__ __forceinline__ float bsum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename I, int EPL>
__device__ __forceinline__ void load_vec(const I *p, float (&x)[EPL]) {
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] = tof(p[e]);
}

// the two float4 pieces of this lane's slice of a D-vector (row of S, k or q) as four pairs
template <int LPR>
__device__ __forceinline__ void load_slice(const float *p, int j, float2 *x) {
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const float4 t = *reinterpret_cast<const float4 *>(p + 4 * (m * LPR + j));
    x[2 * m] = make_float2(t.x, t.y);
    x[2 * m + 1] = make_float2(t.z, t.w);
  }
}

}  // namespace

// at most 64 registers, so that four CTAs (32 warps) share an SM
template <typename I, int D>
__global__ void __launch_bounds__(WARPS * 32, 4) recurrent_kernel(RecArgs a) {
  constexpr int LPR = D / FPL;  // lanes per row group: 16 (d = 128) or 8 (d = 64)
  constexpr int R = D / 32;     // rows per lane: 4 or 2 (LPR = 4 R)
  constexpr int EPL = D / 32;   // staging: features per lane
  const int nh = blockIdx.x, H = a.H, n = nh / H, h = nh % H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % LPR;                     // this lane's place in its group
  const int rg = warp * 8 + (lane / LPR) * R;   // its group's first row within the CTA
  const int rowc = blockIdx.y * RPC;            // the CTA's first state row
  const size_t sbase = ((size_t)nh * D + rowc + rg) * D;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const I *q = static_cast<const I *>(a.q);
  const I *k = static_cast<const I *>(a.k);
  const I *v = static_cast<const I *>(a.v);
  I *o = static_cast<I *>(a.o);
  // the token inputs of TB tokens at a time, staged in shared memory with k normalised and q scaled once
  // per CTA (not once per warp), so that the token loop reads them at shared-memory latency
  __shared__ __align__(16) float ks[TB][D], qs[TB][D], vs[TB][RPC];
  __shared__ __align__(16) float4 gs[TB];  // alpha, beta, k . q

  float2 s[R][4];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (a.S_in) {
      load_slice<LPR>(a.S_in + sbase + (size_t)i * D, j, s[i]);
    } else {
#pragma unroll
      for (int p = 0; p < 4; ++p) s[i][p] = make_float2(0.f, 0.f);
    }
  }

  for (int t0 = 0; t0 < a.T; t0 += TB) {
    const int nt = min(TB, a.T - t0);
    // ---- stage tokens t0 .. t0 + nt - 1: warp w takes tokens w, w + 8 (k, q, their norms, k . q and the
    // gates); every thread a few of the CTA's v entries
    for (int tt = warp; tt < nt; tt += WARPS) {
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
      float kq = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float ke = kk[e] * km, qe = qq[e] * qm;
        ks[tt][lane * EPL + e] = ke;
        qs[tt][lane * EPL + e] = qe;
        kq = fmaf(ke, qe, kq);
      }
      kq = bsum(kq);
      if (lane == 0) gs[tt] = make_float4(expf(a.g[tok]), a.beta[tok], kq, 0.f);
    }
    for (int i = threadIdx.x; i < nt * RPC; i += blockDim.x) {
      const int tt = i / RPC, r = i % RPC;
      vs[tt][r] = tof(v[(((size_t)n * a.T + t0 + tt) * H + h) * D + rowc + r]);
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const float4 gi = gs[tt];
      const float alpha = gi.x, bt = gi.y, kq = gi.z;
      float2 kk[4], qq[4];
      load_slice<LPR>(ks[tt], j, kk);
      load_slice<LPR>(qs[tt], j, qq);
      // this lane's parts of (S k)_i and (S q)_i for its R rows: val[2 i] and val[2 i + 1]
      float val[2 * R];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        float2 pa = __fmul2_rn(s[i][0], kk[0]), pb = __fmul2_rn(s[i][0], qq[0]);
#pragma unroll
        for (int p = 1; p < 4; ++p) {
          pa = __ffma2_rn(s[i][p], kk[p], pa);
          pb = __ffma2_rn(s[i][p], qq[p], pb);
        }
        val[2 * i] = pa.x + pa.y;
        val[2 * i + 1] = pb.x + pb.y;
      }
      // transposed butterfly over the group: each halving step keeps half of the values (the rows selected
      // by that lane bit, from the group's top bit down to bit 2, then S k / S q by bit 1), bit 0 completes
      // the sum; lanes 4i .. 4i + 3 end with row i's two sums
#pragma unroll
      for (int off = LPR / 2, cnt = 2 * R; off >= 2; off >>= 1, cnt >>= 1) {
        const bool hi = (j & off) != 0;
#pragma unroll
        for (int t = 0; t < cnt / 2; ++t)
          val[t] = (hi ? val[cnt / 2 + t] : val[t]) + __shfl_xor_sync(0xffffffffu, hi ? val[t] : val[cnt / 2 + t], off);
      }
      float x = val[0] + __shfl_xor_sync(0xffffffffu, val[0], 1);
      const float y = __shfl_xor_sync(0xffffffffu, x, 2);
      const bool isq = (j & 2) != 0;
      const float dk = isq ? y : x, dq = isq ? x : y;
      const int ri = j >> 2;  // the row whose sums this lane holds
      const float u = bt * (vs[tt][rg + ri] - alpha * dk);
      if ((j & 3) == 0)
        o[(((size_t)n * a.T + t0 + tt) * H + h) * D + rowc + rg + ri] = fromf<I>(fmaf(alpha, dq, u * kq));
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const float ui = __shfl_sync(0xffffffffu, u, (lane & ~(LPR - 1)) + 4 * i);
        const float2 u2 = make_float2(ui, ui);
#pragma unroll
        for (int p = 0; p < 4; ++p) s[i][p] = __ffma2_rn(a2, s[i][p], __fmul2_rn(u2, kk[p]));
      }
    }
    __syncthreads();  // the staged block is read before the next one overwrites it
  }

#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int m = 0; m < 2; ++m)
      *reinterpret_cast<float4 *>(a.S_out + sbase + (size_t)i * D + 4 * (m * LPR + j)) =
          make_float4(s[i][2 * m].x, s[i][2 * m].y, s[i][2 * m + 1].x, s[i][2 * m + 1].y);
}

int launch_recurrent(const RecArgs &a, bool is_bf16, int D, int NH, cudaStream_t st) {
  if (NH == 0) return 0;
  const dim3 grid(NH, D / RPC);
  if (is_bf16 && D == 128) recurrent_kernel<bf16, 128><<<grid, WARPS * 32, 0, st>>>(a);
  else if (is_bf16 && D == 64) recurrent_kernel<bf16, 64><<<grid, WARPS * 32, 0, st>>>(a);
  else if (!is_bf16 && D == 128) recurrent_kernel<float, 128><<<grid, WARPS * 32, 0, st>>>(a);
  else if (!is_bf16 && D == 64) recurrent_kernel<float, 64><<<grid, WARPS * 32, 0, st>>>(a);
  else return -1;
  return (int)cudaGetLastError();
}

}  // namespace gdn
