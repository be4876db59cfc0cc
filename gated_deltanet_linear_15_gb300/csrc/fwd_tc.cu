// Blackwell-native fused forward (bf16 inputs, d = 128): TMA tile loads,
// tcgen05.mma with every accumulator in tensor memory (TMEM), the recurrent
// state resident in TMEM for the whole segment.
//
// Every chunk product is an M = 128 MMA with the feature dimension on the
// TMEM lanes (transposed where that is what puts d = 128 on M):
//   [K; Q] K^T     -> N = strict_tril(K K^T) (rows 0-63), Q K^T (rows 64-127)
//   W^T = K^T X1^T, U^T = V^T X2^T      X1 = Ahat diag(beta), X2 = diag(gp) Ahat diag(beta rgp)
//   Ut^T = U^T - S0 W^T (negated-A MMA accumulating on U^T),   O^T = S0 Qg^T
//   S   = gam_C S0 + Ut^T Kc                Kc = diag(cdec) K (MN-major operand)
//   O^T += Ut^T P^T                         P = diag(gp) tril_incl(Q K^T) diag(rgp)
// with Qg = diag(gam) Q, W^T's columns scaled by gam at read-out, and
// Ahat = (I + diag(beta) N)^{-1} computed on CUDA cores in fp32 (onedev.kr
// FlashQLA talk summary, paragraph on the WY representation for the four
// steps; paragraph on SFU load for pulling the diagonal gamma scaling out of
// the inverse).  Operands are fp16 in 128-byte-swizzled shared memory (see
// umma.cuh); the state is kept in fp32 in TMEM and copied to fp16 once per
// chunk as the operand of the next products.
//
// One CTA of 256 threads per (segment, head); thread 0 issues TMA and MMA,
// both warpgroups read TMEM (each covers lanes 0-127) and do the CUDA-core
// work.  Inputs of chunk c+1 are loaded by TMA while chunk c is computed.
#include "chunk_common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

using namespace umma;

namespace {

constexpr int D = 128;
constexpr int HT = 8192;  // one 64 x 64 fp16 half-tile, 128B-swizzled

// TMEM columns
constexpr uint32_t TM_S = 0, TM_KQ = 128, TM_W = 192, TM_U = 256, TM_O = 320, TM_COLS = 512;

struct __align__(1024) TcSmem {
  // input ring, 2 stages: [K0 | Q0 | K1 | Q1 | V0 | V1] half-tiles (0/1 = feature block)
  uint8_t ring[2][6 * HT];
  uint8_t kc[2 * HT];   // diag(cdec) K        (MN-major B operand: rows = token)
  uint8_t qg[2 * HT];   // diag(gam) Q          (K-major B operand: rows = token)
  uint8_t x1[HT], x2[HT], p[HT];
  uint8_t wu[2 * HT];   // W^T (MN-major B, rows = d_k), later Ut^T (K-major A, rows = d_v)
  uint8_t s0[4 * HT];   // S0 fp16 (K-major A: rows = d_v, two k-blocks of 128 rows)
  float nf[CH * (CH + 4)];
  float g[2][CH], beta[2][CH];  // per ring stage
  Gates gt[2];  // per ring stage; the next chunk's gates are computed during this chunk
  float ys[1152];
  uint64_t bar_tma[2];
  uint64_t bar_mma;
  uint32_t tmem_base;
};

constexpr int LN = CH + 4;

__device__ __forceinline__ uint32_t u32(const void *p) { return smem_u32(p); }

// store 8 fp32 values as one 16-byte fp16 chunk
__device__ __forceinline__ void st_chunk_f16(uint8_t *dst, const float *v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(h);
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1)
    fwd_tc_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ unsigned char smraw[];
  TcSmem &sm = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);

  const int s = blockIdx.x, h = blockIdx.y, role = blockIdx.z;
  const int H = a.H;
  const int n = a.plan.seg_seq[s];
  if (n < 0) return;
  const int j = s - a.plan.seq_seg0[n], nseg = a.plan.seq_nseg[n];
  const int len = a.plan.seq_len[n], chunk0 = a.plan.seq_chunk0[n];
  const int bos = a.plan.seq_bos[n];
  const int nchunks = (len + CH - 1) / CH;
  const int cbeg = j * a.Lseg, cend = min(cbeg + a.Lseg, nchunks);
  const bool window = !(a.flags & kFlagWindowOff);
  int w = 0;
  const int mode = fwd_start_mode(a.gsum, H, h, chunk0, cbeg, j, window, &w);
  bool transition = false;
  if (a.pass == 0) {
    if (j >= nseg - 1) return;
    int w2;
    if (fwd_start_mode(a.gsum, H, h, chunk0, cend, j + 1, window, &w2) != START_FIXUP) return;
    if (role == 1) {
      if (mode != START_FIXUP) return;
      transition = true;
    }
  } else if (role != 0) {
    return;
  }
  const bool outputs = (a.pass == 1);
  const bool states = (a.pass == 2);
  const bool need_v = !transition;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;                      // warpgroup 0 / 1
  const int row = ((warp & 3) << 5) | lane;      // TMEM lane this thread reads
  const size_t DD = (size_t)D * D;
  const size_t sh_idx = (size_t)s * H + h;
  int cfirst = cbeg;
  if (mode == START_WARMUP && !transition) cfirst = cbeg - w;

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    mbar_init(u32(&sm.bar_tma[0]), 1);
    mbar_init(u32(&sm.bar_tma[1]), 1);
    mbar_init(u32(&sm.bar_mma), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmq);
  }
  if (warp == 0) {
    tmem_alloc(u32(&sm.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = sm.tmem_base;
  const uint32_t tm_lane = (uint32_t)((warp & 3) * 32) << 16;

  auto issue_tma = [&](int c, int stage) {
    const int tok0 = bos + c * CH;
    const bool wq = outputs && c >= cbeg;
    const uint32_t bytes = (2 + (wq ? 2 : 0) + (need_v ? 2 : 0)) * HT;
    const uint32_t bar = u32(&sm.bar_tma[stage]);
    uint8_t *st = sm.ring[stage];
    mbar_expect_tx(bar, bytes);
    tma_load_3d(u32(st + 0 * HT), &tmk, 0, h, tok0, bar);
    tma_load_3d(u32(st + 2 * HT), &tmk, 64, h, tok0, bar);
    if (wq) {
      tma_load_3d(u32(st + 1 * HT), &tmq, 0, h, tok0, bar);
      tma_load_3d(u32(st + 3 * HT), &tmq, 64, h, tok0, bar);
    }
    if (need_v) {
      tma_load_3d(u32(st + 4 * HT), &tmv, 0, h, tok0, bar);
      tma_load_3d(u32(st + 5 * HT), &tmv, 64, h, tok0, bar);
    }
  };
  auto issue_gb = [&](int c, int stage, bool with_g) {  // cp.async of (g and) beta for chunk c
    const int tok0 = bos + c * CH;
    const int nvalid = min(CH, len - c * CH);
    if (with_g) load_scalars(sm.g[stage], a.g, H, h, tok0, nvalid, 0);
    load_scalars(sm.beta[stage], a.beta, H, h, tok0, nvalid, 64);
    cp_async_commit();
  };
  if (tid == 0 && cfirst < cend) issue_tma(cfirst, 0);
  if (cfirst < cend) issue_gb(cfirst, 0, true);

  // ---------------------------------------------------------------- initial state -> TMEM
  {
    const float *src = nullptr;
    if (!transition) {
      if (mode == START_INIT) src = a.S0 ? a.S0 + ((size_t)n * H + h) * DD : nullptr;
      else if (mode == START_FIXUP && a.pass != 0) src = a.Sstart + sh_idx * DD;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c0 = wg * 64 + half * 32;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = c0 + i;
        v[i] = src ? src[(size_t)row * D + col] : (transition && col == row ? 1.f : 0.f);
      }
      tmem_st32(tm + tm_lane + TM_S + c0, v);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  int *err = a.status;
  uint32_t mma_phase = 0;
  bool failed = false;
  auto mma_wait = [&]() {
    const bool ok = mbar_wait(u32(&sm.bar_mma), mma_phase, err, 4);
    mma_phase ^= 1;
    fence_after();
    return ok;
  };

  for (int c = cfirst; c < cend && !failed; ++c) {
    const int it = c - cfirst;
    const int stage = it & 1;
    const bool emit = outputs && c >= cbeg;
    const int tok0 = bos + c * CH;
    const int nvalid = min(CH, len - c * CH);
    uint8_t *st = sm.ring[stage];

    float *gbeta = sm.beta[stage];
    float gnext0 = 0.f, gnext1 = 0.f;  // next chunk's log-gates (warp 0), consumed while MMA 4 runs
    if (warp == 0 && c + 1 < cend) {
      const int tokn = bos + (c + 1) * CH, nvn = min(CH, len - (c + 1) * CH);
      if (lane < nvn) gnext0 = a.g[(size_t)(tokn + lane) * H + h];
      if (lane + 32 < nvn) gnext1 = a.g[(size_t)(tokn + lane + 32) * H + h];
    }
    // g, beta of this chunk (issued one chunk ahead) must have landed before the next prefetch reuses cp.async
    cp_async_wait_all();
    // prefetch the next chunk into the other stage (its previous contents were consumed)
    if (tid == 0 && c + 1 < cend) issue_tma(c + 1, stage ^ 1);
    if (c + 1 < cend) issue_gb(c + 1, stage ^ 1, false);
    const bool tma_ok = mbar_wait(u32(&sm.bar_tma[stage]), (it >> 1) & 1, err, 8);
    if (__syncthreads_or(!tma_ok)) {
      failed = true;
      break;
    }
    Gates &G = sm.gt[stage];
    if (it == 0 && warp == 0) {  // later chunks' gates were computed one chunk ahead
      if (gate_prefix(sm.g[stage], G) && lane == 0 && err) atomicOr(err, 1);
    }
    __syncthreads();

    // ---- prep: bf16 -> fp16 in place, L2 norm of q/k rows, Kc = cdec*K, Qg = gam*Q; rows >= nvalid zeroed.
    // Thread t: half-row t of K (t < 128) or of Q (t >= 128): 64 features = one 128-byte swizzled row, the
    // two halves of a row in adjacent lanes (one shuffle for the squared norm); plus quarter-row t of V.
    {
      const bool isq = tid >= 128;
      if (!isq || emit) {
        const int r = (tid >> 1) & 63, hb = tid & 1;
        uint8_t *rowp = st + (isq ? HT : 0) + hb * 2 * HT + r * 128;
        uint32_t raw[32];
#pragma unroll
        for (int chk = 0; chk < 8; ++chk) {
          const uint4 q4 = *reinterpret_cast<const uint4 *>(rowp + ((chk ^ (r & 7)) * 16));
          raw[4 * chk] = q4.x;
          raw[4 * chk + 1] = q4.y;
          raw[4 * chk + 2] = q4.z;
          raw[4 * chk + 3] = q4.w;
        }
        float mul = isq ? a.scale : 1.f;
        if (l2) {
          float ss = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float lo = __uint_as_float(raw[i] << 16), hi = __uint_as_float(raw[i] & 0xffff0000u);
            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
          }
          ss += __shfl_xor_sync(0xffffffffu, ss, 1);
          mul *= rsqrtf(ss + 1e-6f);
        }
        if (r >= nvalid) mul = 0.f;
        const float m2 = mul * (isq ? G.gam[r] : G.cdec[r]);
        uint8_t *row2 = (isq ? sm.qg : sm.kc) + hb * HT + r * 128;
#pragma unroll
        for (int chk = 0; chk < 8; ++chk) {
          uint32_t y[4], z[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t w = raw[4 * chk + i];
            const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
            const __half2 a2 = __floats2half2_rn(lo * mul, hi * mul);
            const __half2 b2 = __floats2half2_rn(lo * m2, hi * m2);
            y[i] = *reinterpret_cast<const uint32_t *>(&a2);
            z[i] = *reinterpret_cast<const uint32_t *>(&b2);
          }
          const int off = (chk ^ (r & 7)) * 16;
          *reinterpret_cast<uint4 *>(rowp + off) = make_uint4(y[0], y[1], y[2], y[3]);
          *reinterpret_cast<uint4 *>(row2 + off) = make_uint4(z[0], z[1], z[2], z[3]);
        }
      }
      if (need_v) {  // quarter-row: 4 chunks of V
        const int r = tid >> 2, qr = tid & 3;
        uint8_t *rowp = st + 4 * HT + (qr >> 1) * HT + r * 128;
        const float mul = r < nvalid ? 1.f : 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int chk = (qr & 1) * 4 + cc;
          uint4 q4 = *reinterpret_cast<const uint4 *>(rowp + ((chk ^ (r & 7)) * 16));
          uint32_t *w = reinterpret_cast<uint32_t *>(&q4);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 a2 = __floats2half2_rn(__uint_as_float(w[i] << 16) * mul,
                                                 __uint_as_float(w[i] & 0xffff0000u) * mul);
            w[i] = *reinterpret_cast<const uint32_t *>(&a2);
          }
          *reinterpret_cast<uint4 *>(rowp + ((chk ^ (r & 7)) * 16)) = q4;
        }
      }
    }
    fence_async_smem();
    __syncthreads();

    // ---- MMA 1: [K; Q] K^T  (M = 128, N = 64, K = 128)
    if (tid == 0) {
      fence_after();
      const uint32_t idesc = idesc_f16(128, 64, false, false);
      const uint32_t base = u32(st);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
        mma_f16(tm + TM_KQ, sdesc(base + koff, 16, 1024), sdesc(base + koff, 16, 1024), idesc, kk > 0);
      }
      mma_commit(u32(&sm.bar_mma));
    }
    __syncwarp();
    if (__syncthreads_or(!mma_wait())) {
      failed = true;
      break;
    }

    // ---- read-out: N (fp32, rows 0-63) and P (fp16, rows 64-127); each warpgroup takes 32 columns
    if (row < 64 || emit) {
      float v[32];
      const int c0 = wg * 32;
      tmem_ld32(tm + tm_lane + TM_KQ + c0, v);
      if (row < 64) {
#pragma unroll
        for (int i = 0; i < 32; ++i) sm.nf[row * LN + c0 + i] = v[i];
      } else {
        const int r = row - 64;
        const float gr = G.gp[r];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int col = c0 + q4 * 8 + i;
            y[i] = col <= r ? v[q4 * 8 + i] * gr * G.rgp[col] : 0.f;
          }
          const int chk = (c0 >> 3) + q4;
          st_chunk_f16(sm.p + r * 128 + ((chk ^ (r & 7)) * 16), y);
        }
      }
    }
    fence_before();
    __syncthreads();

    // ---- Ahat (fp32 diagonal blocks, TF32 tensor-core merges) -> X1, X2 (fp16, K-major: rows = r)
    wy_inverse<false, false>(sm.nf, LN, gbeta, sm.ys, [&](int r, int c, float a0, float a1) {
      const float b0 = gbeta[c], b1 = gbeta[c + 1], gr = G.gp[r];
      const uint32_t off = sw128_offset(r, c);
      *reinterpret_cast<__half2 *>(sm.x1 + off) = __floats2half2_rn(a0 * b0, a1 * b1);
      *reinterpret_cast<__half2 *>(sm.x2 + off) =
          __floats2half2_rn(c <= r ? a0 * b0 * (gr * G.rgp[c]) : 0.f,
                            c + 1 <= r ? a1 * b1 * (gr * G.rgp[c + 1]) : 0.f);
    });

    // ---- MMA 2: W^T = K^T X1^T, U^T = V^T X2^T  (M = 128, N = 64, K = 64)
    if (tid == 0) {
      fence_after();
      const uint32_t idesc = idesc_f16(128, 64, true, false);
      const uint32_t kb = u32(st), vb = u32(st + 4 * HT), x1b = u32(sm.x1), x2b = u32(sm.x2);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_f16(tm + TM_W, sdesc(kb + kk * 2048, 2 * HT, 1024), sdesc(x1b + kk * 32, 16, 1024), idesc, kk > 0);
      }
      if (need_v) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tm + TM_U, sdesc(vb + kk * 2048, HT, 1024), sdesc(x2b + kk * 32, 16, 1024), idesc, kk > 0);
      }
      mma_commit(u32(&sm.bar_mma));
    }
    __syncwarp();
    // meanwhile: S0 -> fp16 operand copy, gam_C * S0 back into TMEM (state copy for the backward)
    {
      const float gC = G.gamC;
      f16 *stg = states && c >= cbeg
                     ? static_cast<f16 *>(a.states) + ((size_t)(chunk0 + c) * H + h) * DD + (size_t)row * D
                     : nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c0 = wg * 64 + half * 32;
        float v[32];
        tmem_ld32(tm + tm_lane + TM_S + c0, v);
        const int kb = c0 >> 6;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chk = ((c0 & 63) >> 3) + q4;
          uint8_t *dst = sm.s0 + kb * 2 * HT + row * 128 + ((chk ^ (row & 7)) * 16);
          st_chunk_f16(dst, v + q4 * 8);
          if (stg) *reinterpret_cast<uint4 *>(stg + c0 + q4 * 8) = *reinterpret_cast<const uint4 *>(dst);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gC;
        tmem_st32(tm + tm_lane + TM_S + c0, v);
      }
    }
    if (__syncthreads_or(!mma_wait())) {
      failed = true;
      break;
    }

    // ---- W^T read-out: columns scaled by gam -> fp16 MN-major B (rows = d_k)
    {
      const int c0 = wg * 32;
      float v[32];
      tmem_ld32(tm + tm_lane + TM_W + c0, v);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = v[q4 * 8 + i] * G.gam[c0 + q4 * 8 + i];
        const int chk = (c0 >> 3) + q4;
        st_chunk_f16(sm.wu + row * 128 + ((chk ^ (row & 7)) * 16), y);
      }
    }
    fence_before();
    fence_async_smem();
    __syncthreads();

    // ---- MMA 3: Ut^T = U^T - S0 W^T;  O^T = S0 Qg^T   (M = 128, N = 64, K = 128)
    if (tid == 0) {
      fence_after();
      const uint32_t s0b = u32(sm.s0), wb = u32(sm.wu), qb = u32(sm.qg);
      const uint32_t id_u = idesc_f16(128, 64, false, true, /*neg_a=*/true);
      const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
        mma_f16(tm + TM_U, sdesc(s0b + aoff, 16, 1024), sdesc(wb + kk * 2048, 2 * HT, 1024), id_u,
                need_v || kk > 0);
      }
      if (emit) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * HT + (kk & 3) * 32;
          mma_f16(tm + TM_O, sdesc(s0b + aoff, 16, 1024), sdesc(qb + boff, 16, 1024), id_o, kk > 0);
        }
      }
      mma_commit(u32(&sm.bar_mma));
    }
    __syncwarp();
    if (__syncthreads_or(!mma_wait())) {
      failed = true;
      break;
    }

    // ---- Ut^T read-out -> fp16 K-major A (rows = d_v, k = token)
    {
      const int c0 = wg * 32;
      float v[32];
      tmem_ld32(tm + tm_lane + TM_U + c0, v);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int chk = (c0 >> 3) + q4;
        st_chunk_f16(sm.wu + row * 128 + ((chk ^ (row & 7)) * 16), v + q4 * 8);
      }
    }
    fence_before();
    fence_async_smem();
    __syncthreads();

    // ---- MMA 4: S += Ut^T Kc (N = 128, K = 64);  O^T += Ut^T P^T (N = 64, K = 64)
    if (tid == 0) {
      fence_after();
      const uint32_t ub = u32(sm.wu), kcb = u32(sm.kc), pb = u32(sm.p);
      const uint32_t id_s = idesc_f16(128, 128, false, true);
      const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16(tm + TM_S, sdesc(ub + kk * 32, 16, 1024), sdesc(kcb + kk * 2048, HT, 1024), id_s, true);
      if (emit) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tm + TM_O, sdesc(ub + kk * 32, 16, 1024), sdesc(pb + kk * 32, 16, 1024), id_o, true);
      }
      mma_commit(u32(&sm.bar_mma));
    }
    __syncwarp();
    if (warp == 0 && c + 1 < cend) {  // gates of the next chunk, overlapping MMA 4
      float *gn = sm.g[stage ^ 1];
      gn[lane] = gnext0;
      gn[lane + 32] = gnext1;
      __syncwarp();
      if (gate_prefix(gn, sm.gt[stage ^ 1]) && lane == 0 && err) atomicOr(err, 1);
    }
    if (__syncthreads_or(!mma_wait())) {
      failed = true;
      break;
    }

    // ---- O^T read-out -> bf16 [token][d_v] staging in qg (free now) -> coalesced rows of o
    if (emit) {
      const int c0 = wg * 32;
      float v[32];
      tmem_ld32(tm + tm_lane + TM_O + c0, v);
      bf16 *stg = reinterpret_cast<bf16 *>(sm.qg);
#pragma unroll
      for (int i = 0; i < 32; ++i) stg[(c0 + i) * D + row] = __float2bfloat16_rn(v[i]);
    }
    fence_before();
    __syncthreads();
    if (emit) {
      const uint4 *stg = reinterpret_cast<const uint4 *>(sm.qg);
      bf16 *og = static_cast<bf16 *>(a.o);
      for (int e = tid; e < CH * (D / 8); e += NTHREADS) {
        const int r = e >> 4, cc = e & 15;
        if (r < nvalid) *reinterpret_cast<uint4 *>(og + ((size_t)(tok0 + r) * H + h) * D + cc * 8) = stg[e];
      }
    }
  }

  // ---------------------------------------------------------------- end-of-segment state
  if (!failed) {
    float *dst = nullptr;
    if (a.pass == 0) dst = (transition ? a.Mbuf : a.Ebuf) + sh_idx * DD;
    else if (j == nseg - 1 && a.ST) dst = a.ST + ((size_t)n * H + h) * DD;
    if (dst) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c0 = wg * 64 + half * 32;
        float v[32];
        tmem_ld32(tm + tm_lane + TM_S + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4 *>(dst + (size_t)row * D + c0 + 4 * q4) =
              make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
      }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tm, TM_COLS);
}

size_t fwd_tc_smem_bytes() { return sizeof(TcSmem) + 1024; }

int launch_fwd_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                  cudaStream_t st) {
  const size_t smem = fwd_tc_smem_bytes();
  static_assert(sizeof(TcSmem) + 1024 <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  fwd_tc_kernel<<<grid, NTHREADS, smem, st>>>(a, tq, tk, tv);
  return (int)cudaGetLastError();
}

}  // namespace gdn
