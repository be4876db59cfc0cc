// WY tiles of every (chunk, head) for the backward (bf16, d = 128), computed once
// and read by the three backward kernels instead of each re-deriving them:
//   Ahat = (I + diag(beta) N)^{-1},  N = strict_tril(K^ K^T)   (K^ the normalised keys)
//   X1   = Ahat diag(beta)
//   X2   = diag(gp) Ahat diag(beta rgp)   (lower triangle incl. the diagonal)
// as fp16 [64][64] row-major tiles, three per (chunk, head) (onedev.kr FlashQLA
// talk summary, paragraph on the WY representation; the inverse itself is the
// blocked doubling of chunk_common.cuh).  The arithmetic is the one the fused
// kernels run inline: fp16 keys normalised with the same rsqrt, fp32 Gram
// matrix, fp32 inverse with TF32 tensor-core merges, one rounding to fp16.
//
// One CTA of 256 threads per (chunk, head), ~41 KB of shared memory (several
// CTAs per SM); N on the legacy mma.sync path (a 64 x 64 x 128 product).
#include "chunk_common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int D = 128;
constexpr int LDK = D + 8;  // padded fp16 row (ldmatrix without bank conflicts)
constexpr int LN = CH + 4;

struct WySmem {
  f16 k[CH * LDK];
  float nf[CH * LN];
  float g[CH], beta[CH];
  Gates gt;
  float ys[1152];
};

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 4) wy_kernel(WyArgs a) {
  extern __shared__ __align__(128) unsigned char smraw[];
  WySmem &sm = *reinterpret_cast<WySmem *>(smraw);
  const int gc = blockIdx.x, h = blockIdx.y, H = a.H;
  const int n = a.plan.chunk_seq[gc];
  if (n < 0) return;
  const int lc = gc - a.plan.seq_chunk0[n];
  const long tok0 = (long)a.plan.seq_bos[n] + (long)lc * CH;
  const int nvalid = min(CH, a.plan.seq_len[n] - lc * CH);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;

  load_tile<bf16, D>(sm.k, LDK, static_cast<const bf16 *>(a.k), H, h, tok0, nvalid);
  load_scalars(sm.g, a.g, H, h, tok0, nvalid, 0);
  load_scalars(sm.beta, a.beta, H, h, tok0, nvalid, 64);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  if (warp == 0 && gate_prefix(sm.g, sm.gt) && lane == 0 && a.status) atomicOr(a.status, 1);
  {  // K^ in place: thread t takes quarter-row t (32 features), the four quarters in adjacent lanes
    const int r = tid >> 2, qq = tid & 3;
    uint4 *row4 = reinterpret_cast<uint4 *>(sm.k + r * LDK + qq * 32);  // 64 bytes, 16-byte aligned
    uint4 raw[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) raw[c] = row4[c];
    const uint32_t *w = reinterpret_cast<const uint32_t *>(raw);
    float x[32];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      ss = fmaf(x[2 * i], x[2 * i], fmaf(x[2 * i + 1], x[2 * i + 1], ss));
    }
    float mul = 1.f;
    if (l2) {
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      mul = rsqrtf(ss + 1e-6f);
    }
    if (r >= nvalid) mul = 0.f;
    uint32_t y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const __half2 h2 = __floats2half2_rn(x[2 * i] * mul, x[2 * i + 1] * mul);
      y[i] = *reinterpret_cast<const uint32_t *>(&h2);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) row4[c] = make_uint4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
  }
  __syncthreads();
  if (warp < 4) {  // N = K^ K^T, 32 x 32 blocks; only the strict lower triangle is read later
    Acc<32, 32> acc;
    acc.zero();
    const int m0 = (warp >> 1) * 32, n0 = (warp & 1) * 32;
    warp_mma<32, 32, false, false>(acc, sm.k, LDK, sm.k, LDK, m0, n0, D);
    acc.each([&](int r, int c, float &v) { sm.nf[(m0 + r) * LN + n0 + c] = v; });
  }
  __syncthreads();
  f16 *tiles = static_cast<f16 *>(a.wy) + ((size_t)gc * H + h) * 3 * CH * CH;
  wy_inverse<false, false>(sm.nf, LN, sm.beta, sm.ys, [&](int r, int c, float a0, float a1) {
    const float2 bb = *reinterpret_cast<const float2 *>(sm.beta + c), rg = *reinterpret_cast<const float2 *>(sm.gt.rgp + c);
    const float gr = sm.gt.gp[r], x0 = a0 * bb.x, x1 = a1 * bb.y;
    const size_t off = (size_t)r * CH + c;
    *reinterpret_cast<__half2 *>(tiles + off) = __floats2half2_rn(x0, x1);
    *reinterpret_cast<__half2 *>(tiles + CH * CH + off) =
        __floats2half2_rn(c <= r ? x0 * (gr * rg.x) : 0.f, c + 1 <= r ? x1 * (gr * rg.y) : 0.f);
    *reinterpret_cast<__half2 *>(tiles + 2 * CH * CH + off) = __floats2half2_rn(a0, a1);
  });
}

int launch_wy(const WyArgs &a, int CH_max, cudaStream_t st) {
  if (CH_max == 0) return 0;
  const size_t smem = sizeof(WySmem);
  cudaError_t e = cudaFuncSetAttribute(wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  wy_kernel<<<dim3(CH_max, a.H), NTHREADS, smem, st>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace gdn
