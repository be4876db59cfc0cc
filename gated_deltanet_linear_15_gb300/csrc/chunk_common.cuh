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
// receives the norm of each row.  Returns true when one of this thread's values
// does not fit an fp16 operand (numeric guard; always false for fp32 operands).
template <typename I, typename E, int D>
__device__ __forceinline__ bool prep_rows(E *t, int ld, float mul, bool l2, float *norm_out) {
  static_assert(sizeof(I) == sizeof(E), "in-place conversion needs equal element sizes");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const I *src = reinterpret_cast<const I *>(t);
  bool bad = false;
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
    for (int i = 0; i < D / 32; ++i) {
      if (std::is_same<E, f16>::value) bad |= f16_out(x[i] * f);
      t[r * ld + lane + 32 * i] = fromf<E>(x[i] * f);
    }
  }
  return bad;
}

// Gate quantities of one chunk from the raw log-gates g[0..CH) (one warp).
//   G_r   = sum_{i<=r} g_i                 (in-chunk inclusive prefix)
//   gam_r = exp(G_r)                       (decay from the chunk start)
//   gp_r  = exp(G_r - G_mid), rgp_r = exp(G_mid - G_r)   (gamma factoring, centred)
//   cdec_r = exp(G_last - G_r)             (decay from token r to the chunk end)
// Each exponential is taken once per token (onedev.kr FlashQLA talk summary,
// paragraph on SFU load: the diagonal scaling is pulled out of the inverse).
// The decay ratio gamma_r / gamma_c (c <= r) is then gp_r * rgp_c.  The pages
// put no lower bound on alpha in (0, 1) (same page, paragraph on the effective
// sliding window), so a chunk can decay by more than fp32 can factor: when
// |G_r - G_mid| exceeds FACTOR_RANGE for some r, gp or rgp would overflow and
// the chunk is marked `pw`; its ratios are then taken pairwise as
// exp(G_r - G_c) (C^2 / 2 exponentials, for that chunk only).  Log-gates below
// GATE_FLOOR are raised to it: exp(GATE_FLOOR) and every ratio across such a
// token are zero in fp32 either way, and the prefix sums keep their precision.
// A chunk whose prefix sums stay within |G| <= 16 takes them in plain fp32
// (their differences then carry an absolute error of a few 1e-6).  A chunk
// that decays further can hold a large decay (|G| ~ 100) followed by slow
// decay, where plain fp32 prefix sums lose the small differences that the
// ratios need; it carries the sums as unevaluated pairs hi + lo of fp32 values
// (each addition error-free by Knuth's TwoSum) and forms each exponent argument
// (a difference of two prefix sums) from both parts.  (fp64 would do the same,
// but it is slow on this part.)
struct __align__(16) Gates {
  float Ghi[CH], Glo[CH];
  float gam[CH], gp[CH], rgp[CH], cdec[CH];
  float gamC;  // exp(G_last)
  float Glog;  // G_last, the chunk's summed log-gates
  int pw;      // nonzero: take decay ratios pairwise (the span leaves the factoring range)
};

// (hi, lo) += (bh, bl), hi + lo exact up to lo's rounding (Knuth's TwoSum, then a renormalisation)
__device__ __forceinline__ void two_add(float &hi, float &lo, float bh, float bl) {
  const float s = hi + bh, v = s - hi;
  const float e = (hi - (s - v)) + (bh - v);
  const float l = lo + bl + e;
  hi = s + l;
  lo = l - (hi - s);
}
// (ah + al) - (bh + bl) as one fp32 value
__device__ __forceinline__ float two_diff(float ah, float al, float bh, float bl) { return (ah - bh) + (al - bl); }

// gamma_r / gamma_c for c <= r (callers mask c > r themselves); the pairwise form out of line, so that
// the factored one stays small in the kernels' read-out loops
static __device__ __noinline__ float gratio_pw(const Gates &gt, int r, int c) {
  return expf(two_diff(gt.Ghi[r], gt.Glo[r], gt.Ghi[c], gt.Glo[c]));
}
__device__ __forceinline__ float gratio(const Gates &gt, int r, int c) {
  return gt.pw ? gratio_pw(gt, r, c) : gt.gp[r] * gt.rgp[c];
}
// the ratios for columns c, c + 1 (c even) of row r, one check for both
__device__ __forceinline__ float2 gratio2(const Gates &gt, int r, int c) {
  if (!gt.pw) {
    const float2 rg = *reinterpret_cast<const float2 *>(gt.rgp + c);
    const float gr = gt.gp[r];
    return make_float2(gr * rg.x, gr * rg.y);
  }
  return make_float2(gratio_pw(gt, r, c), gratio_pw(gt, r, c + 1));
}

// 16 consecutive floats from 16-byte aligned shared memory (four vector loads)
__device__ __forceinline__ void ld16f(const float *p, float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 t = reinterpret_cast<const float4 *>(p)[q];
    v[4 * q] = t.x;
    v[4 * q + 1] = t.y;
    v[4 * q + 2] = t.z;
    v[4 * q + 3] = t.w;
  }
}

// The in-chunk prefix sums and decay factors of a chunk (lane l of the calling warp holds the log-gates of
// tokens l and l + 32), written for the tokens of `halves` (bit 0: tokens 0-31, bit 1: tokens 32-63); the
// bit-0 writer also sets gamC and pw.  Every caller forms the full scans, so two warps can split the
// exponentials (one half each) with no exchange; returns pw.
__device__ __forceinline__ bool gate_prefix_part(float ga, float gb, Gates &gt, int halves) {
  const int lane = threadIdx.x & 31;
  ga = fmaxf(ga, GATE_FLOOR);
  gb = fmaxf(gb, GATE_FLOOR);
  float a = ga, b = gb, al = 0.f, bl = 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) {
      a += ya;
      b += yb;
    }
  }
  float Gm = __shfl_sync(0xffffffffu, a, 31), Gml = 0.f;
  b += Gm;
  // |G| over the chunk: beyond 16, redo the sums as hi + lo pairs (a warp-uniform branch)
  if (__any_sync(0xffffffffu, fmaxf(fabsf(a), fabsf(b)) > 16.f)) {
    a = ga;
    b = gb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float ya = __shfl_up_sync(0xffffffffu, a, o), yal = __shfl_up_sync(0xffffffffu, al, o);
      const float yb = __shfl_up_sync(0xffffffffu, b, o), ybl = __shfl_up_sync(0xffffffffu, bl, o);
      if (lane >= o) {
        two_add(a, al, ya, yal);
        two_add(b, bl, yb, ybl);
      }
    }
    Gm = __shfl_sync(0xffffffffu, a, 31);
    Gml = __shfl_sync(0xffffffffu, al, 31);
    two_add(b, bl, Gm, Gml);
  }
  const float Gl = __shfl_sync(0xffffffffu, b, 31), Gll = __shfl_sync(0xffffffffu, bl, 31);
  const float da = two_diff(a, al, Gm, Gml), db = two_diff(b, bl, Gm, Gml);
  if (halves & 1) {
    gt.Ghi[lane] = a;
    gt.Glo[lane] = al;
    gt.gam[lane] = expf(a + al);
    gt.gp[lane] = expf(da);
    gt.rgp[lane] = expf(-da);
    gt.cdec[lane] = expf(two_diff(Gl, Gll, a, al));
    if (lane == 0) {
      gt.gamC = expf(Gl + Gll);
      gt.Glog = Gl + Gll;
    }
  }
  if (halves & 2) {
    gt.Ghi[lane + 32] = b;
    gt.Glo[lane + 32] = bl;
    gt.gam[lane + 32] = expf(b + bl);
    gt.gp[lane + 32] = expf(db);
    gt.rgp[lane + 32] = expf(-db);
    gt.cdec[lane + 32] = expf(two_diff(Gl, Gll, b, bl));
  }
  float rng = fmaxf(fabsf(da), fabsf(db));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rng = fmaxf(rng, __shfl_xor_sync(0xffffffffu, rng, o));
  const bool pw = rng > FACTOR_RANGE;
  if ((halves & 1) && lane == 0) gt.pw = pw;
  return pw;
}
// one warp, both halves, log-gates from shared memory
__device__ __forceinline__ bool gate_prefix(const float *g, Gates &gt) {
  const int lane = threadIdx.x & 31;
  return gate_prefix_part(g[lane], g[lane + 32], gt, 3);
}

// o[i] = gamma_r / gamma_{cb + i} for cb + i <= r, 0 above the diagonal (eight columns from cb, a multiple of 8),
// with the form chosen at compile time: read-out loops are instantiated once per form and pick one by Gates::pw,
// so the factored loop carries none of the pairwise code
template <bool PW> __device__ __forceinline__ void ratio8(const Gates &gt, int r, int cb, float (&o)[8]) {
  if constexpr (!PW) {
    const float4 a = reinterpret_cast<const float4 *>(gt.rgp + cb)[0], b = reinterpret_cast<const float4 *>(gt.rgp + cb)[1];
    const float gr = gt.gp[r];
    o[0] = gr * a.x; o[1] = gr * a.y; o[2] = gr * a.z; o[3] = gr * a.w;
    o[4] = gr * b.x; o[5] = gr * b.y; o[6] = gr * b.z; o[7] = gr * b.w;
  } else {
    const float Gr = gt.Ghi[r], Grl = gt.Glo[r];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = cb + i <= r ? expf(two_diff(Gr, Grl, gt.Ghi[cb + i], gt.Glo[cb + i])) : 0.f;
  }
}
// The ratios at the eight entries of a 16 x 16 fragment that one lane holds (rows ra, ra + 8; columns ta,
// ta + 1, ta + 8, ta + 9; ta even): o[4x + 2h + e] = gamma_{ra + 8h} / gamma_{ta + 8x + e}.  The factored form
// does not zero the entries above the diagonal (the callers mask them); the pairwise form does.
template <bool PW> __device__ __forceinline__ void ratio_frag(const Gates &gt, int ra, int ta, float (&o)[8]) {
  if constexpr (!PW) {
    const float2 a = *reinterpret_cast<const float2 *>(gt.rgp + ta), b = *reinterpret_cast<const float2 *>(gt.rgp + ta + 8);
    const float g0 = gt.gp[ra], g1 = gt.gp[ra + 8];
    o[0] = g0 * a.x; o[1] = g0 * a.y; o[2] = g1 * a.x; o[3] = g1 * a.y;
    o[4] = g0 * b.x; o[5] = g0 * b.y; o[6] = g1 * b.x; o[7] = g1 * b.y;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = ra + 8 * ((i >> 1) & 1), c = ta + 8 * (i >> 2) + (i & 1);
      o[i] = c <= r ? expf(two_diff(gt.Ghi[r], gt.Glo[r], gt.Ghi[c], gt.Glo[c])) : 0.f;
    }
  }
}
// the same with the form chosen at run time (the pairwise form element by element out of line)
__device__ __forceinline__ void gratio8(const Gates &gt, int r, int cb, float (&o)[8]) {
  if (!gt.pw) {
    const float4 a = reinterpret_cast<const float4 *>(gt.rgp + cb)[0], b = reinterpret_cast<const float4 *>(gt.rgp + cb)[1];
    const float gr = gt.gp[r];
    o[0] = gr * a.x; o[1] = gr * a.y; o[2] = gr * a.z; o[3] = gr * a.w;
    o[4] = gr * b.x; o[5] = gr * b.y; o[6] = gr * b.z; o[7] = gr * b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = cb + i <= r ? gratio_pw(gt, r, cb + i) : 0.f;
  }
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

// Ahat = (I + diag(beta) N)^{-1} for the strictly lower N held in `nf` (row
// stride ldn; only its strict lower triangle is read, the strict upper
// triangle serves as scratch).  The four diagonal 16 x 16 blocks are inverted
// by forward substitution (one column per lane) into `dinv` (>= 64 x 17
// floats); the off-diagonal part follows in two doubling levels of the block
// identity  [[A, 0], [C, B]]^{-1} = [[A^-1, 0], [-B^-1 C A^-1, B^-1]]:  16 -> 32
// (blocks (1,0) and (3,2)) and 32 -> 64 (the lower-left 32 x 32 block), each a
// pair of m16n8k8 TF32 tensor-core products (3xTF32 when PRECISE).  Every
// element of Ahat is then handed to out(r, c, Ahat[r][c], Ahat[r][c + 1]) once
// (c even), the zero upper blocks only when with_zeros; with NF_T the strict
// lower part is also stored transposed into
// the strict upper triangle of nf.  Uses warps 0-7 (any further warps only join
// the barriers, or, with WARPS8, do not take part at all); ends with a proxy
// fence and a barrier.
template <bool PRECISE, bool NF_T, bool WARPS8 = false, class Out>
__device__ __forceinline__ void wy_inverse(float *nf, int ldn, const float *beta, float *dinv, Out out,
                                           bool with_zeros = true) {
  // WARPS8: called by warps 0-7 only, which synchronise among themselves (named barrier 1)
  auto bar = [] {
    if (WARPS8) asm volatile("bar.sync 1, 256;\n" ::: "memory");
    else __syncthreads();
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int DL = 17;  // dinv row stride
  if (warp < 4 && lane < 16) {  // column jj of block warp; rows of N read as 16-byte vectors (broadcast)
    const int b = warp * 16, jj = lane;
    float x[16], bt[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 t = *reinterpret_cast<const float4 *>(beta + b + 4 * q);
      bt[4 * q] = t.x;
      bt[4 * q + 1] = t.y;
      bt[4 * q + 2] = t.z;
      bt[4 * q + 3] = t.w;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < (r + 3) / 4; ++q) {
        const float4 n4 = *reinterpret_cast<const float4 *>(nf + (b + r) * ldn + b + 4 * q);
        const float nv[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (4 * q + u < r) acc[u] = fmaf(nv[u], x[4 * q + u], acc[u]);
      }
      x[r] = ((r == jj) ? 1.f : 0.f) - bt[r] * ((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
    // stored only now, so that no store sits between the row loads above (dinv may alias nf)
#pragma unroll
    for (int r = 0; r < 16; ++r) dinv[(b + r) * DL + jj] = x[r];
  }
  bar();
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
  // fragment coordinates (m16n8k8): A element i at (gr + 8 (i & 1), gc + 4 (i >> 1)),
  // B element h at (k = gc + 4 h, n = gr), accumulator e at (gr + 8 (e >> 1), 2 gc + (e & 1))
  const int gr = lane >> 2, gc = lane & 3;
  // level 1: X_{I,J} = -D_I (T_IJ D_J) for (I, J) = (1, 0), (3, 2); warp w < 4: pair w / 2, columns 8 (w % 2)..
  // The result stays in registers (x1v) for the hand-out and goes, transposed, to the scratch slot
  // nf[(16 J + c) * ldn + 16 I + r] for level 2.  (dinv is exactly zero above each block's diagonal.)
  float x1v[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp < 4) {
    const int I = 2 * (warp >> 1) + 1, J = I - 1, nt = warp & 1;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    const float b0 = beta[16 * I + gr], b1 = beta[16 * I + gr + 8];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int k0 = 16 * J + 8 * ks;
      const float av[4] = {b0 * nf[(16 * I + gr) * ldn + k0 + gc], b1 * nf[(16 * I + gr + 8) * ldn + k0 + gc],
                           b0 * nf[(16 * I + gr) * ldn + k0 + gc + 4], b1 * nf[(16 * I + gr + 8) * ldn + k0 + gc + 4]};
      const float bv[2] = {dinv[(k0 + gc) * DL + 8 * nt + gr], dinv[(k0 + gc + 4) * DL + 8 * nt + gr]};
      mma(y, av, bv);
    }
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int a0 = 16 * I;
      const float av[4] = {dinv[(a0 + gr) * DL + 8 * ks + gc], dinv[(a0 + gr + 8) * DL + 8 * ks + gc],
                           dinv[(a0 + gr) * DL + 8 * ks + gc + 4], dinv[(a0 + gr + 8) * DL + 8 * ks + gc + 4]};
      float bv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // B element (k = 8 ks + gc + 4 h, n = gr) from the accumulator y
        const int src = (gc + 4 * h) * 4 + (gr >> 1);
        const float e0 = __shfl_sync(0xffffffffu, y[2 * ks + 0], src);
        const float e1 = __shfl_sync(0xffffffffu, y[2 * ks + 1], src);
        bv[h] = (gr & 1) ? e1 : e0;
      }
      mma(x1v, av, bv);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x1v[e] = -x1v[e];
      const int r = gr + 8 * (e >> 1), c = 8 * nt + 2 * gc + (e & 1);
      nf[(16 * J + c) * ldn + 16 * I + r] = x1v[e];
    }
  }
  bar();
  // level 2: Y = T_LL E0 (32 x 32, stored transposed in the upper-right quadrant), then X_LL = -E1 Y;
  // warp (mt, nt) owns the m16n8 tile at rows 16 mt, columns 8 nt.  Block relations are warp-uniform.
  const int mt = (warp >> 2) & 1, nt = warp & 3;
  if (warp < 8) {
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    const int ra = 32 + 16 * mt;
    const float b0 = beta[ra + gr], b1 = beta[ra + gr + 8];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (ks < nt) continue;  // E0[k][j] = 0 for k < j
      const int k0 = 8 * ks;
      const float av[4] = {b0 * nf[(ra + gr) * ldn + k0 + gc], b1 * nf[(ra + gr + 8) * ldn + k0 + gc],
                           b0 * nf[(ra + gr) * ldn + k0 + gc + 4], b1 * nf[(ra + gr + 8) * ldn + k0 + gc + 4]};
      float bv[2];
      if ((ks >> 1) == (nt >> 1)) {  // E0 diagonal block
        bv[0] = dinv[(k0 + gc) * DL + ((8 * nt + gr) & 15)];
        bv[1] = dinv[(k0 + gc + 4) * DL + ((8 * nt + gr) & 15)];
      } else {  // E0 block (1, 0): level-1 scratch
        bv[0] = nf[(8 * nt + gr) * ldn + k0 + gc];
        bv[1] = nf[(8 * nt + gr) * ldn + k0 + gc + 4];
      }
      mma(y, av, bv);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // Y[i][j] -> nf[j * ldn + 32 + i]
      const int i = 16 * mt + gr + 8 * (e >> 1), j = 8 * nt + 2 * gc + (e & 1);
      nf[j * ldn + 32 + i] = y[e];
    }
  }
  bar();
  float xl[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp < 8) {
    const int a0 = 32 + 16 * mt;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (ks > 2 * mt + 1) continue;  // E1[i][k] = 0 for k > i
      const int k0 = 32 + 8 * ks;
      float av[4];
      if ((ks >> 1) == mt) {  // E1 diagonal block
        av[0] = dinv[(a0 + gr) * DL + ((k0 + gc) & 15)];
        av[1] = dinv[(a0 + gr + 8) * DL + ((k0 + gc) & 15)];
        av[2] = dinv[(a0 + gr) * DL + ((k0 + gc + 4) & 15)];
        av[3] = dinv[(a0 + gr + 8) * DL + ((k0 + gc + 4) & 15)];
      } else {  // E1 block (3, 2): level-1 scratch
        av[0] = nf[(k0 + gc) * ldn + a0 + gr];
        av[1] = nf[(k0 + gc) * ldn + a0 + gr + 8];
        av[2] = nf[(k0 + gc + 4) * ldn + a0 + gr];
        av[3] = nf[(k0 + gc + 4) * ldn + a0 + gr + 8];
      }
      const float bv[2] = {nf[(8 * nt + gr) * ldn + k0 + gc], nf[(8 * nt + gr) * ldn + k0 + gc + 4]};
      mma(xl, av, bv);
    }
  }
  bar();  // Y is read; its slots may now take the transposed lower-left block
  if (warp < 8) {
    auto give = [&](int r, int c, float a0, float a1) {
      out(r, c, a0, a1);
      if (NF_T) {
        if (c < r) nf[c * ldn + r] = a0;
        if (c + 1 < r) nf[(c + 1) * ldn + r] = a1;
      }
    };
    // lower-left 32 x 32 (registers of every warp)
#pragma unroll
    for (int h = 0; h < 2; ++h) give(32 + 16 * mt + gr + 8 * h, 8 * nt + 2 * gc, -xl[2 * h], -xl[2 * h + 1]);
    // blocks (1, 0) and (3, 2) (registers of warps 0-3)
    if (warp < 4) {
      const int I = 2 * (warp >> 1) + 1, nt1 = warp & 1;
#pragma unroll
      for (int h = 0; h < 2; ++h) give(16 * I + gr + 8 * h, 16 * (I - 1) + 8 * nt1 + 2 * gc, x1v[2 * h], x1v[2 * h + 1]);
    }
    // diagonal blocks from dinv: thread t -> block t / 64, rows (t % 64) / 4 and columns 2 (t % 4) + {0, 8}
    {
      const int t = threadIdx.x, blk = t >> 6, r = (t & 63) >> 2, cc = 2 * (t & 3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = cc + 8 * h;
        give(16 * blk + r, 16 * blk + c, dinv[(16 * blk + r) * DL + c], dinv[(16 * blk + r) * DL + c + 1]);
      }
    }
    // zeros: the six 16 x 16 blocks above the diagonal (768 pairs, three per thread); a caller whose
    // output tiles keep them from an earlier call passes with_zeros = false
#pragma unroll
    for (int i = 0; i < 3 && with_zeros; ++i) {
      const int pidx = threadIdx.x + 256 * i;  // pair index
      const int b = pidx >> 7, w = pidx & 127;   // block 0..5, pair within block
      const int bi = b < 3 ? 0 : (b < 5 ? 1 : 2);
      const int bj = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
      out(16 * bi + (w >> 3), 16 * bj + 2 * (w & 7), 0.f, 0.f);
    }
  }
  umma_fence_proxy();  // shared-memory operands written above are read by the tensor-core async proxy
  bar();
}

}  // namespace gdn
