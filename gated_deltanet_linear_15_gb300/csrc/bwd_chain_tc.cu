// Blackwell-native reverse state chain of the chunked backward (bf16 inputs,
// d = 128): one CTA per (segment, head), chunks in reverse order, dS (the
// gradient w.r.t. a chunk's end state) resident in fp32 TMEM.  The forward's
// chunk context supplies the operand forms of K and Q (normalised, fp16),
// P = diag(gp) tril(Q K^T) diag(rgp) and the gam-scaled W^T of every chunk
// (TMA, with dO), so a chunk is dO's conversion and two tensor-core rounds:
//   Y = dS K^T, Z = dO^T P, dS += (diag(gam) dO)^T Q;   dUt^T = Y diag(cdec) + Z (read-out)
//   dS <- dS - dUt^T W                                    (after gam_C dS and the fp16 copy)
// and the fp16 dS at every chunk end and the chunk's fp16 dUt^T (the operand of
// round 2, which the local-gradient kernel would otherwise recompute from dS, K,
// dO and P) go to the workspace by TMA store for the local-gradient kernel.  Pass 0 (reverse sequence parallelism) runs a
// segment from zero (role 0) or the transition from I with dO = 0 (role 1);
// pass 1 runs it from its exact end gradient and stores the per-chunk dS
// (and dS0 for the first segment).  Layouts and primitives as in fwd_tc.cu.
#include "chunk_common.cuh"
#include "fixup.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

using namespace umma;

namespace {

constexpr int D = 128;
constexpr int HT = 8192;
constexpr uint32_t TM_S = 0, TM_DU = 256, TM_Y = 320, TM_COLS = 512;

struct __align__(1024) ChainTcSmem {
  // input ring, 2 stages: [K0 | Q0 | K1 | Q1 | dO0 | dO1 | P | W0 W1] half-tiles (0/1 = feature block;
  // K, Q the fp16 operand tiles of the context; W = the gam-scaled W^T tile [d_k][token])
  uint8_t ring[2][9 * HT];
  uint8_t kc[2 * HT];       // dUt^T (K-major A, rows = d_v)
  uint8_t dog[2 * HT];      // diag(gam) dO (MN-major A, rows = token)
  uint8_t ds16[4 * HT];     // dS fp16 (K-major A: rows = d_v, two k-blocks of 128 rows)
  float g[2][CH];
  Gates gt[2];
  uint64_t bar_tma[2];
  uint64_t bar_mma;
  uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t u32(const void *p) { return smem_u32(p); }

__device__ __forceinline__ void st_chunk_f16(uint8_t *dst, const float *v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(h);
}

}  // namespace

// One work item: segment s of head h in pass `pass` (0: pass A, role 0 the start gradient from zero or its
// warm-up, role 1 the reverse transition; 1: the per-chunk dS).  A CTA may run several items in turn: the
// first that does work allocates the TMEM columns (have_tm), which the caller frees after the last one.
__device__ __forceinline__ void chain_tc_item(const BwdArgs &a, const CUtensorMap &tm3, const CUtensorMap &tmdo,
                                              const CUtensorMap &tmp, const CUtensorMap &tmw, const CUtensorMap &tmds,
                                              const CUtensorMap &tmdu, int s, int h, int role, int pass,
                                              bool &have_tm) {
  extern __shared__ unsigned char smraw[];
  ChainTcSmem &sm =
      *reinterpret_cast<ChainTcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  // pass A of a call in which no segment needs the exact fix-up (status[2], set by the fix-up mode scan)
  if (pass == 0 && a.status && a.status[2] == 0) return;
  const int H = a.H;
  const int n = a.plan.seg_seq[s];
  if (n < 0) return;
  const int j = s - a.plan.seq_seg0[n], nseg = a.plan.seq_nseg[n];
  const int len = a.plan.seq_len[n], chunk0 = a.plan.seq_chunk0[n];
  const int bos = a.plan.seq_bos[n];
  const int nchunks = (len + CH - 1) / CH;
  const int cbeg = seg_begin(j, a.Lfirst, a.Lseg), cend = min(seg_begin(j + 1, a.Lfirst, a.Lseg), nchunks);
  const bool window = !(a.flags & kFlagWindowOff);
  int w = 0;
  const int mode = bwd_start_mode(a.gsum, H, h, chunk0, cend, nchunks, j, nseg, window, &w);
  bool transition = false;
  if (pass == 0) {
    if (j == 0) return;
    int w2;
    if (bwd_start_mode(a.gsum, H, h, chunk0, cbeg, nchunks, j - 1, nseg, window, &w2) != START_FIXUP) return;
    if (role == 1) {
      if (mode != START_FIXUP) return;
      transition = true;
    }
  } else if (role != 0) {
    return;
  }
  if (a.flags & kFlagDebugWaitTimeout) {  // test hook: an expiring bounded wait, then return
    __shared__ uint64_t dbg_bar;
    if (threadIdx.x == 0) debug_expire_wait(&dbg_bar, a.status, 4);
    return;
  }
  const bool store = (pass == 1);
  const bool with_do = !transition;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;
  const int row = ((warp & 3) << 5) | lane;
  const size_t DD = (size_t)D * D;
  const size_t sh_idx = (size_t)s * H + h;
  int clast = cend - 1;
  if (mode == START_WARMUP && !transition) clast = cend - 1 + w;

  if (tid == 0) {
    mbar_init(u32(&sm.bar_tma[0]), 1);
    mbar_init(u32(&sm.bar_tma[1]), 1);
    mbar_init(u32(&sm.bar_mma), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tma_prefetch_desc(&tm3);
    tma_prefetch_desc(&tmdo);
    tma_prefetch_desc(&tmp);
    tma_prefetch_desc(&tmw);
    if (store) {
      tma_prefetch_desc(&tmds);
      tma_prefetch_desc(&tmdu);
    }
  }
  if (!have_tm && warp == 0) {
    tmem_alloc(u32(&sm.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  have_tm = true;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = sm.tmem_base;
  const uint32_t tl = (uint32_t)((warp & 3) * 32) << 16;

  auto issue_tma = [&](int c, int stage) {
    const int tok0 = bos + c * CH;
    const int crow = (chunk0 + c) * H + h;  // (chunk, head) index of the context tiles
    const uint32_t bar = u32(&sm.bar_tma[stage]);
    uint8_t *st = sm.ring[stage];
    const int qrow = crow * TQ_TILES * CH;
    mbar_expect_tx(bar, (4 + (with_do ? 5 : 0)) * HT);
    tma_load_3d(u32(st + 0 * HT), &tm3, 0, qrow + TQ_K * CH, 0, bar);
    tma_load_3d(u32(st + 2 * HT), &tm3, 64, qrow + TQ_K * CH, 0, bar);
    tma_load_3d(u32(st + 7 * HT), &tmw, 0, (crow * T128_TILES + T128_W) * D, 0, bar);
    if (with_do) {
      tma_load_3d(u32(st + 1 * HT), &tm3, 0, qrow + TQ_Q * CH, 0, bar);
      tma_load_3d(u32(st + 3 * HT), &tm3, 64, qrow + TQ_Q * CH, 0, bar);
      tma_load_3d(u32(st + 4 * HT), &tmdo, 0, h, tok0, bar);
      tma_load_3d(u32(st + 5 * HT), &tmdo, 64, h, tok0, bar);
      tma_load_3d(u32(st + 6 * HT), &tmp, 0, (crow * T64_TILES + T64_P) * CH, 0, bar);
    }
  };
  if (clast >= cbeg) {
    if (tid == NTHREADS) issue_tma(clast, 0);
    load_scalars(sm.g[0], a.g, H, h, bos + clast * CH, min(CH, len - clast * CH), 0);
    cp_async_commit();
  }

  // initial dS -> TMEM
  {
    const float *src = nullptr;
    if (!transition) {
      if (mode == START_INIT) src = a.dST ? a.dST + ((size_t)n * H + h) * DD : nullptr;
      else if (mode == START_FIXUP && pass != 0) src = a.dSend + sh_idx * DD;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      if (warp >= NWARPS) break;  // the producer warp holds no state
      const int c0 = wg * 64 + half * 32;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = c0 + i;
        v[i] = src ? __ldcg(src + (size_t)row * D + col) : (transition && col == row ? 1.f : 0.f);
      }
      tmem_st32(tm + tl + TM_S + c0, v);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  int *err = a.status;
  uint32_t mma_phase = 0;
  bool failed = false;
  bool nbad = false;  // numeric guard: an fp16 operand out of range
  auto mma_wait = [&]() {
    const bool ok = mbar_wait(u32(&sm.bar_mma), mma_phase, err, 4);
    mma_phase ^= 1;
    fence_after();
    return ok;
  };

  // Lane 0 of warp NWARPS (the producer) issues every TMA copy and tensor-core product (an MMA issue
  // blocks its thread while the tensor pipe's queue is full; the nine tile loads of a chunk cost its
  // thread ~1.5 k cycles); the 8 worker warps convert dO, copy dS and read TMEM.  The two sides meet at
  // CTA-wide OR-barriers B2 (dO and the dS copy ready: round 1) and B3 (dUt^T ready: round 2), which
  // carry a failed wait; the workers sync among themselves on barrier 1, and the producer tells them
  // that the previous chunk's dS store has read ds16 (barrier 2, arrive / sync).  A worker that gives up
  // at barrier 1 releases the producer with one CTA-wide OR-barrier.
  const bool producer = warp == NWARPS;
  bool release = false;
  for (int c = clast; c >= cbeg; --c) {
    const int it = clast - c;
    const int stage = it & 1;
    const int nvalid = min(CH, len - c * CH);
    uint8_t *st = sm.ring[stage];
    if (producer) {
      // ================================================================ producer
      if (lane == 0) {
        // round 2 of the previous chunk (the second of two commits per chunk: parity 1) has read its
        // ring stage, which takes the tiles of chunk c - 1 below
        if (it > 0) mbar_wait(u32(&sm.bar_mma), 1, err, 4);
        if (store) tma_store_wait_read();  // the previous chunk's dS and dUt^T stores have read ds16 and kc
      }
      __syncwarp();
      named_bar_arrive<2, NTHREADS + 32>();
      if (lane == 0 && c - 1 >= cbeg) issue_tma(c - 1, stage ^ 1);
      __syncwarp();
      if (__syncthreads_or(false)) {  // B2: dO and the fp16 dS copy are ready
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        if (store && c < cend) {  // the fp16 dS at the end of chunk c and its fp16 dO, for the local-gradient kernel
          const int srow = ((chunk0 + c) * H + h) * D;
          tma_store_3d(&tmds, 0, srow, 0, u32(sm.ds16));
          tma_store_3d(&tmds, 64, srow, 0, u32(sm.ds16 + 2 * HT));
          tma_store_3d(&tmdu, 0, (((chunk0 + c) * H + h) * TC_TILES + TC_DO) * D, 0, u32(st + 4 * HT));
          tma_store_commit();
        }
        const uint32_t id_kk = idesc_f16(128, 64, false, false);
        const uint32_t id_mm = idesc_f16(128, 64, true, true);
        const uint32_t dsb = u32(sm.ds16), kb = u32(st), dob = u32(st + 4 * HT), pb = u32(st + 6 * HT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 2 * HT + (kk & 3) * 32;
          mma_f16s(tm + TM_Y, sdesc_s(dsb, 16, 1024) + (off), sdesc_s(kb, 16, 1024) + (off), id_kk, kk > 0);
        }
        if (with_do) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16s(tm + TM_DU, sdesc_s(dob, HT, 1024) + (kk * 2048), sdesc_s(pb, HT, 1024) + (kk * 2048), id_mm,
                     kk > 0);
          const uint32_t id_s = idesc_f16(128, 128, true, true), dgb = u32(sm.dog), qb = u32(st + HT);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16s(tm + TM_S, sdesc_s(dgb, HT, 1024) + (kk * 2048), sdesc_s(qb, 2 * HT, 1024) + (kk * 2048), id_s,
                     true);
        }
        mma_commit(u32(&sm.bar_mma));
      }
      __syncwarp();
      if (__syncthreads_or(false)) {  // B3: dUt^T is ready
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        const uint32_t id_kk_neg = idesc_f16(128, 128, false, false, true);
        const uint32_t dub = u32(sm.kc), wb = u32(st + 7 * HT);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16s(tm + TM_S, sdesc_s(dub, 16, 1024) + (kk * 32), sdesc_s(wb, 16, 1024) + (kk * 32), id_kk_neg, true);
        mma_commit(u32(&sm.bar_mma));
        if (store && c < cend) {  // dUt^T of chunk c for the local-gradient kernel (read before the next
                                  // chunk's read-out rewrites kc)
          tma_store_3d(&tmdu, 0, (((chunk0 + c) * H + h) * TC_TILES + TC_DUT) * D, 0, dub);
          tma_store_commit();
        }
      }
      __syncwarp();
      continue;
    }

    // ================================================================ workers
    float gnext0 = 0.f, gnext1 = 0.f;  // log-gates of the next (previous in time) chunk, warps 0 and 1
    if (warp < 2 && c - 1 >= cbeg) {
      const int tokn = bos + (c - 1) * CH, nvn = min(CH, len - (c - 1) * CH);
      if (lane < nvn) gnext0 = a.g[(size_t)(tokn + lane) * H + h];
      if (lane + 32 < nvn) gnext1 = a.g[(size_t)(tokn + lane + 32) * H + h];
    }
    if (it == 0) cp_async_wait_all();  // the first chunk's gates; later ones come from gnext
    {
      const bool tma_ok = mbar_wait(u32(&sm.bar_tma[stage]), (it >> 1) & 1, err, 8);
      uint32_t any;
      asm volatile(
          "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
          : "=r"(any)
          : "r"((uint32_t)(!tma_ok || failed)), "n"(NTHREADS)
          : "memory");
      if (any) {
        failed = release = true;
        break;
      }
    }
    Gates &G = sm.gt[stage];
    if (it == 0) {
      if (warp == 0) gate_prefix(sm.g[stage], G);
      named_bar_sync<1, NTHREADS>();
    }

    // ---- prep: dO -> fp16 in place and diag(gam) dO (rows >= nvalid zero); K, Q come as operand tiles
    if (with_do) {
      const int r = tid >> 2, qr = tid & 3;
      uint8_t *rowp = st + 4 * HT + (qr >> 1) * HT + r * 128;
      uint8_t *rowg = sm.dog + (qr >> 1) * HT + r * 128;
      const float mul = r < nvalid ? 1.f : 0.f, mg = mul * G.gam[r];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int off = (((qr & 1) * 4 + cc) ^ (r & 7)) * 16;
        uint4 q4 = *reinterpret_cast<const uint4 *>(rowp + off);
        uint4 g4;
        uint32_t *wv = reinterpret_cast<uint32_t *>(&q4), *gv = reinterpret_cast<uint32_t *>(&g4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __uint_as_float(wv[i] << 16), hi = __uint_as_float(wv[i] & 0xffff0000u);
          nbad |= f16_out(lo * mul) | f16_out(hi * mul);
          const __half2 a2 = __floats2half2_rn(lo * mul, hi * mul), b2 = __floats2half2_rn(lo * mg, hi * mg);
          wv[i] = *reinterpret_cast<const uint32_t *>(&a2);
          gv[i] = *reinterpret_cast<const uint32_t *>(&b2);
        }
        *reinterpret_cast<uint4 *>(rowp + off) = q4;
        *reinterpret_cast<uint4 *>(rowg + off) = g4;
      }
    }
    named_bar_sync<2, NTHREADS + 32>();  // the previous chunk's stores have read ds16 and kc
    // ---- dS (end of chunk c) -> fp16 operand copy, gam_C dS back into TMEM
    {
      const float gC = G.gamC;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c0 = wg * 64 + half * 32;
        float v[32];
        tmem_ld32(tm + tl + TM_S + c0, v);
        const int kb = c0 >> 6;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chk = ((c0 & 63) >> 3) + q4;
          st_chunk_f16(sm.ds16 + kb * 2 * HT + row * 128 + ((chk ^ (row & 7)) * 16), v + q4 * 8);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          nbad |= f16_out(v[i]);
          v[i] *= gC;
        }
        tmem_st32(tm + tl + TM_S + c0, v);
      }
    }
    fence_async_smem();
    fence_before();
    if (__syncthreads_or(false)) {  // B2: the producer stores dS and issues round 1
      failed = true;
      break;
    }
    failed |= !mma_wait();  // round 1
    {  // dUt^T = Y diag(cdec) + Z -> fp16 K-major A (rows = d_v, k = token)
      const int c0 = wg * 32;
      float y[32], v[32];
      tmem_ld32(tm + tl + TM_Y + c0, y);
      if (with_do) {
        tmem_ld32(tm + tl + TM_DU + c0, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 ca = reinterpret_cast<const float4 *>(G.cdec + c0 + q4 * 8)[0];
        const float4 cb = reinterpret_cast<const float4 *>(G.cdec + c0 + q4 * 8)[1];
        const float cd[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[q4 * 8 + i] = fmaf(cd[i], y[q4 * 8 + i], v[q4 * 8 + i]);
          nbad |= f16_out(v[q4 * 8 + i]);
        }
        st_chunk_f16(sm.kc + row * 128 + ((((c0 >> 3) + q4) ^ (row & 7)) * 16), v + q4 * 8);
      }
    }
    fence_before();
    fence_async_smem();
    if (__syncthreads_or(failed)) {  // B3: the producer issues round 2
      failed = true;
      break;
    }
    if (warp < 2 && c - 1 >= cbeg)  // gates of the next chunk, overlapping the last product: a half per warp
      gate_prefix_part(gnext0, gnext1, sm.gt[stage ^ 1], 1 << warp);
    failed |= !mma_wait();  // round 2
  }
  if (release) __syncthreads_or(true);  // meet the producer at its pending CTA-wide barrier: it stops there

  if (!failed && warp < NWARPS) {
    float *dst = nullptr;
    if (pass == 0) dst = (transition ? a.Rbuf : a.Fbuf) + sh_idx * DD;
    else if (j == 0 && a.dS0) dst = a.dS0 + ((size_t)n * H + h) * DD;
    if (dst) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c0 = wg * 64 + half * 32;
        float v[32];
        tmem_ld32(tm + tl + TM_S + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4 *>(dst + (size_t)row * D + c0 + 4 * q4) =
              make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
      }
    }
  }
  if (nbad && err) atomicOr(err, 1);
  if (tid == NTHREADS && store) tma_store_wait_all();
  fence_before();
  __syncthreads();
  fence_after();
  if (tid == 0) {  // the next item of this CTA initialises them again
    mbar_inval(u32(&sm.bar_tma[0]));
    mbar_inval(u32(&sm.bar_tma[1]));
    mbar_inval(u32(&sm.bar_mma));
  }
}

// The TMEM columns of the items a CTA ran, once all of them are done.
__device__ __forceinline__ void chain_tc_release(bool have_tm) {
  if (!have_tm) return;
  extern __shared__ unsigned char smraw[];
  ChainTcSmem &sm =
      *reinterpret_cast<ChainTcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  fence_before();
  __syncthreads();
  fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(sm.tmem_base, TM_COLS);
}

template <bool SCHED>
__global__ void __launch_bounds__(NTHREADS + 32, 1)
    bwd_chain_tc_kernel(BwdArgs a, const __grid_constant__ CUtensorMap tm3, const __grid_constant__ CUtensorMap tmdo,
                        const __grid_constant__ CUtensorMap tmp, const __grid_constant__ CUtensorMap tmw,
                        const __grid_constant__ CUtensorMap tmds, const __grid_constant__ CUtensorMap tmdu) {
  pdl_trigger();
  pdl_wait();
  int s = blockIdx.x, h = blockIdx.y, role = blockIdx.z, pass = a.pass;
  int *doneA = nullptr;  // a pass-A item reports its completion here
  bool have_tm = false;
  if (!SCHED && a.bal_pairs > 0 && pass != 0) {
    // balanced chain over equal-length sequences of bal_ns segments each (1-D grid): CTA b < bal_big runs the
    // b-th later segment (j >= 1) of the (sequence, head) pairs, every other CTA a share of the pairs' shorter
    // first segments (pairs k, k + G - bal_big, ...)
    const int ns = a.bal_ns, b = blockIdx.x, G = gridDim.x;
    if (b < a.bal_big) {
      const int pair = b / (ns - 1);
      chain_tc_item(a, tm3, tmdo, tmp, tmw, tmds, tmdu, (pair / a.H) * ns + 1 + b % (ns - 1), pair % a.H, 0, pass,
                    have_tm);
    } else {
      for (int k = b - a.bal_big; k < a.bal_pairs; k += G - a.bal_big)
        chain_tc_item(a, tm3, tmdo, tmp, tmw, tmds, tmdu, (k / a.H) * ns, k % a.H, 0, pass, have_tm);
    }
    chain_tc_release(have_tm);
    return;
  }
  if (!SCHED && pass == 0 && a.passA_items > 0) {
    // pass A by ticket (1-D grid of at most one CTA per SM): item t is role t & 1 of segment (t / 2) % S,
    // head (t / 2) / S (S segments); a call whose segments need no exact fix-up returns at once
    if (a.status && a.status[2] == 0) return;
    const int S = a.passA_items / (2 * a.H);  // segments
    __shared__ int tk;
    for (;;) {
      if (threadIdx.x == 0) tk = atomicAdd(a.status + 5, 1);
      __syncthreads();
      const int t = tk;
      __syncthreads();  // every thread has its ticket before thread 0 takes the next one
      if (t >= a.passA_items) break;
      chain_tc_item(a, tm3, tmdo, tmp, tmw, tmds, tmdu, (t >> 1) % S, (t >> 1) / S, t & 1, 0, have_tm);
    }
    chain_tc_release(have_tm);
    return;
  }
  if (SCHED) {
    // single-launch sequence parallelism: this CTA runs the ticket-th item of the work lists (see Sched)
    __shared__ int tk, ok;
    const Sched &sc = a.sched;
    const int tid = threadIdx.x;
    if (tid == 0) tk = atomicAdd(sc.hdr, 1);
    __syncthreads();
    constexpr int NRB = D / FIX_ROWS;
    const int nA = __ldcg(sc.hdr + 1), nBn = __ldcg(sc.hdr + 2), nF = __ldcg(sc.hdr + 3), nBf = __ldcg(sc.hdr + 4);
    int t = tk;
    if (t < nA) {  // pass A
      const int e = sc.listA[t];
      s = (e >> 1) / a.H;
      h = (e >> 1) % a.H;
      role = e & 1;
      pass = 0;
      doneA = sc.doneA + a.plan.seg_seq[s] * a.H + h;
    } else if ((t -= nA) < nBn) {  // the chain from an end that needs no fix-up
      s = sc.listBn[t] / a.H;
      h = sc.listBn[t] % a.H;
      role = 0;
    } else if ((t -= nBn) < nF * NRB) {  // a fix-up row block, once its (sequence, head)'s pass A is done
      if (tid >= 256) return;
      const int pair = sc.listF[t / NRB];
      if (tid == 0) ok = wait_count_geq(sc.doneA + pair, sc.needA[pair], PEER_WAIT_LIMIT);
      fix_bar();
      if (!ok) {
        if (tid == 0 && a.status) atomicOr(a.status, 16);
        return;
      }
      __threadfence();
      FixupArgs fx;
      fx.ticket = nullptr;
      fx.plan = a.plan;
      fx.gsum = a.gsum;
      fx.E = a.Fbuf;
      fx.M = a.Rbuf;
      fx.out = a.dSend;
      fx.H = a.H;
      fx.D = D;
      fx.Lseg = a.Lseg;
      fx.Lfirst = a.Lfirst;
      fx.flags = a.flags;
      fx.reverse = 1;
      fx.fixflag = nullptr;
      fx.status = a.status;
      extern __shared__ unsigned char smraw[];
      fixup_rows<D>(fx, t % NRB, pair % a.H, pair / a.H,
                    reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023));
      __threadfence();
      fix_bar();
      if (tid == 0) atomicAdd(sc.doneF + pair, 1);
      return;
    } else if ((t -= nF * NRB) < nBf) {  // the chain from a fixed-up end, once its fix-up blocks are done
      s = sc.listBf[t] / a.H;
      h = sc.listBf[t] % a.H;
      role = 0;
      const int pair = a.plan.seg_seq[s] * a.H + h;
      if (tid == 0) {
        const bool hook = (a.flags & kFlagDebugPeerTimeout) != 0;  // test hook: a wait that cannot succeed
        ok = wait_count_geq(sc.doneF + pair, hook ? NRB + 1 : NRB, hook ? 1024 : PEER_WAIT_LIMIT);
        if (!ok && a.status) atomicOr(a.status, 16);
      }
      __syncthreads();
      if (!ok) return;
      __threadfence();
    } else {
      return;  // a ticket past the lists: no work
    }
  }
  chain_tc_item(a, tm3, tmdo, tmp, tmw, tmds, tmdu, s, h, role, pass, have_tm);
  chain_tc_release(have_tm);
  if (doneA) {  // the start-gradient / transition stores of every thread are visible before the count
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(doneA, 1);
  }
}

int launch_bwd_chain_tc(const BwdArgs &a, const CUtensorMap *maps, dim3 grid, cudaStream_t st) {
  const size_t smem = sizeof(ChainTcSmem) + 1024;
  static_assert(sizeof(ChainTcSmem) + 1024 <= 232448 - 256, "shared memory budget (the rest: static shared memory)");
  static_assert(fixup_smem_bytes<D>() <= sizeof(ChainTcSmem), "a fix-up row block fits the kernel's shared memory");
  auto kern = a.sched_on ? bwd_chain_tc_kernel<true> : bwd_chain_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(kern, grid, dim3(NTHREADS + 32), smem, st, a, maps[0], maps[1], maps[2], maps[3], maps[4],
                         maps[5]);
}

}  // namespace gdn
