// Per-chunk building blocks shared by the forward and backward chunk kernels:
// tile loads, in-kernel L2 normalisation, gate prefix sums, and the unit
// lower-triangular inverse of the WY stage.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace gdn {

// Load a CH x D tile of a [tokens, H, D] input tensor (element type I) into a
// shared tile of the same element size: row r = token tok0 + r of head h, rows
// r >= nvalid zero-filled.  The raw input bits land in the tile; prep_rows()
// converts them to the operand type in place.
template <typename I, int D>
__device__ __forceinline__ void load_tile(void *dst, int ld, const I *base, int H, int h, long tok0, int nvalid) {
  constexpr int EPV = 16 / sizeof(I);  // elements per 16-byte piece
  constexpr int VPR = D / EPV;
  I *d = static_cast<I *>(dst);
  for (int e = threadIdx.x; e < CH * VPR; e += NTHREADS) {
    const int r = e / VPR, cidx = e % VPR;
    const bool valid = r < nvalid;
    const I *src = base + ((size_t)(tok0 + (valid ? r : 0)) * H + h) * D + cidx * EPV;
    cp_async16(d + r * ld + cidx * EPV, src, valid);
  }
}

// Load CH scalars x[(tok0 + r) * H + h] (zero for r >= nvalid) into dst[0..CH).
__device__ __forceinline__ void load_scalars(float *dst, const float *base, int H, int h, long tok0, int nvalid,
                                             int thread0) {
  const int r = threadIdx.x - thread0;
  if (r >= 0 && r < CH) {
    const bool valid = r < nvalid;
    cp_async4(dst + r, base + (size_t)(tok0 + (valid ? r : 0)) * H + h, valid);
  }
}

// In place, one warp per row: raw input values x (type I) become operand values
// (type E)  x * mul / sqrt(sum x^2 + 1e-6)  when `l2`, else  x * mul.  The
// normalisation's row reduction uses warp shuffles; `norm_out` (optional)
// receives the norm of each row.
template <typename I, typename E, int D>
__device__ __forceinline__ void prep_rows(E *t, int ld, float mul, bool l2, float *norm_out) {
  static_assert(sizeof(I) == sizeof(E), "in-place conversion needs equal element sizes");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const I *src = reinterpret_cast<const I *>(t);
  for (int r = warp; r < CH; r += NWARPS) {
    float x[D / 32];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      x[i] = tof(src[r * ld + lane + 32 * i]);
      ss += x[i] * x[i];
    }
    float f = mul;
    if (l2) {
      ss = warp_sum(ss);
      const float nrm = sqrtf(ss + 1e-6f);
      f = mul / nrm;
      if (norm_out && lane == 0) norm_out[r] = nrm;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < D / 32; ++i) t[r * ld + lane + 32 * i] = fromf<E>(x[i] * f);
  }
}

// Gate quantities of one chunk from the raw log-gates g[0..CH) (one warp).
//   G_r   = sum_{i<=r} g_i                 (in-chunk inclusive prefix)
//   gam_r = exp(G_r)                       (decay from the chunk start)
//   gp_r  = exp(G_r - G_mid), rgp_r = exp(G_mid - G_r)   (gamma factoring, centred)
//   cdec_r = exp(G_last - G_r)             (decay from token r to the chunk end)
// Each exponential is taken once per token (onedev.kr FlashQLA talk summary,
// paragraph on SFU load: the diagonal scaling is pulled out of the inverse).
// Returns true in lane 0 if |G_r - G_mid| exceeds the factoring range.
struct Gates {
  float G[CH], gam[CH], gp[CH], rgp[CH], cdec[CH];
  float gamC;  // exp(G_last)
};

__device__ __forceinline__ bool gate_prefix(const float *g, Gates &gt) {
  const int lane = threadIdx.x & 31;
  float a = g[lane], b = g[lane + 32];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float ya = __shfl_up_sync(0xffffffffu, a, o);
    const float yb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) {
      a += ya;
      b += yb;
    }
  }
  const float Gmid = __shfl_sync(0xffffffffu, a, 31);
  b += Gmid;
  const float Glast = __shfl_sync(0xffffffffu, b, 31);
  gt.G[lane] = a;
  gt.G[lane + 32] = b;
  gt.gam[lane] = expf(a);
  gt.gam[lane + 32] = expf(b);
  gt.gp[lane] = expf(a - Gmid);
  gt.gp[lane + 32] = expf(b - Gmid);
  gt.rgp[lane] = expf(Gmid - a);
  gt.rgp[lane + 32] = expf(Gmid - b);
  gt.cdec[lane] = expf(Glast - a);
  gt.cdec[lane + 32] = expf(Glast - b);
  if (lane == 0) gt.gamC = expf(Glast);
  float rng = fmaxf(fabsf(a - Gmid), fabsf(b - Gmid));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rng = fmaxf(rng, __shfl_xor_sync(0xffffffffu, rng, o));
  return rng > FACTOR_RANGE;
}

// Ahat entry (a, b) from the transposed upper-triangle storage written by wy_inverse<., true>.
__device__ __forceinline__ float ahat_at(const float *nf, int ldn, int a, int b) {
  return a == b ? 1.f : (a > b ? nf[b * ldn + a] : 0.f);
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
// x ~ hi + lo, both tf32
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// c += a * b with fp32 operands given as values: 3xTF32
__device__ __forceinline__ void mma_3xtf32(float (&c)[4], const float (&a)[4], const float (&b)[2]) {
  uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
#pragma unroll
  for (int i = 0; i < 2; ++i) split_tf32(b[i], bh[i], bl[i]);
  mma_tf32(c, al, bh);
  mma_tf32(c, ah, bl);
  mma_tf32(c, ah, bh);
}

__device__ __forceinline__ void umma_fence_proxy() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

template <bool PRECISE, bool NF_T, class Out>
__device__ __forceinline__ void wy_inverse(float *nf, int ldn, const float *beta, float *dinv, Out out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int DL = 17;  // dinv row stride
  if (warp < 4 && lane < 16) {
    const int b = warp * 16, jj = lane;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) {
        if (i & 1) s1 += nf[(b + r) * ldn + b + i] * x[i];
        else s0 += nf[(b + r) * ldn + b + i] * x[i];
      }
      x[r] = ((r == jj) ? 1.f : 0.f) - beta[b + r] * (s0 + s1);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) dinv[(warp * 16 + r) * DL + jj] = x[r];
  }
  __syncthreads();
  auto mma = [&](float(&c)[4], const float(&av)[4], const float(&bv)[2]) {
    if (PRECISE) {
      mma_3xtf32(c, av, bv);
    } else {
      uint32_t ah[4], bh[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) ah[i] = to_tf32(av[i]);
      bh[0] = to_tf32(bv[0]);
      bh[1] = to_tf32(bv[1]);
      mma_tf32(c, ah, bh);
    }
  };
  if (warp < 8) {  // eight column slices; further warps (if any) only join the barriers
  const int gr = lane >> 2, gc = lane & 3;
  const int J0 = warp >> 1;               // first row block with non-zero entries in this slice
  const int cl = 8 * (warp & 1);          // slice column offset inside block J0
  // B fragment (k = 8*ks + gc (+4), n = gr) of a 16 x 8 block held in accumulator layout
  auto bfrag = [&](const float(&c)[4], int ks, float(&bv)[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int krow = gc + 4 * h;               // row inside the 8-row half ks
      const int src = krow * 4 + (gr >> 1);      // lane holding (row krow (+8 ks), col gr)
      const float e0 = __shfl_sync(0xffffffffu, c[2 * ks + 0], src);
      const float e1 = __shfl_sync(0xffffffffu, c[2 * ks + 1], src);
      bv[h] = (gr & 1) ? e1 : e0;
    }
  };
  float X[4][4];
#pragma unroll
  for (int I = 0; I < 4; ++I)
#pragma unroll
    for (int e = 0; e < 4; ++e) X[I][e] = 0.f;
  // X_J0 = columns of D_J0^{-1}
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int r = gr + 8 * (e >> 1), c = cl + 2 * gc + (e & 1);
#pragma unroll
    for (int I = 0; I < 4; ++I)
      if (I == J0) X[I][e] = dinv[(I * 16 + r) * DL + c];
  }
#pragma unroll
  for (int I = 1; I < 4; ++I) {
    if (I <= J0) continue;
    const int ra = 16 * I + gr;
    const float b0 = beta[ra], b1 = beta[ra + 8];
    float y0[4] = {0.f, 0.f, 0.f, 0.f}, y1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int K = 0; K < 3; ++K) {
      if (K < J0 || K >= I) continue;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const int k0 = 16 * K + 8 * ks;
        const float av[4] = {b0 * nf[ra * ldn + k0 + gc], b1 * nf[(ra + 8) * ldn + k0 + gc],
                             b0 * nf[ra * ldn + k0 + gc + 4], b1 * nf[(ra + 8) * ldn + k0 + gc + 4]};
        float bv[2];
        bfrag(X[K], ks, bv);
        if (ks == 0) mma(y0, av, bv);
        else mma(y1, av, bv);
      }
    }
    float z[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) z[e] = -(y0[e] + y1[e]);
    float x0[4] = {0.f, 0.f, 0.f, 0.f}, x1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int kc = 8 * ks;
      const float av[4] = {dinv[(I * 16 + gr) * DL + kc + gc], dinv[(I * 16 + gr + 8) * DL + kc + gc],
                           dinv[(I * 16 + gr) * DL + kc + gc + 4], dinv[(I * 16 + gr + 8) * DL + kc + gc + 4]};
      float bv[2];
      bfrag(z, ks, bv);
      if (ks == 0) mma(x0, av, bv);
      else mma(x1, av, bv);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) X[I][e] = x0[e] + x1[e];
  }
  // hand out every element of the slice (rows 0..63, columns 8w..8w+7)
#pragma unroll
  for (int I = 0; I < 4; ++I)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = 16 * I + gr + 8 * h, c = 8 * warp + 2 * gc;
      const float a0 = X[I][2 * h], a1 = X[I][2 * h + 1];
      out(r, c, a0, a1);
      if (NF_T) {
        if (c < r) nf[c * ldn + r] = a0;
        if (c + 1 < r) nf[(c + 1) * ldn + r] = a1;
      }
    }
  }
  umma_fence_proxy();  // shared-memory operands written above are read by the tensor-core async proxy
  __syncthreads();
}

}  // namespace gdn
