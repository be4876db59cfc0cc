// Start-state fix-up (forward: S_start[j+1] = S_start[j] M_j + E_j over the segments of one (sequence,
// head); the reverse chain mirrors it with the segment ends), the sequential composition of the segment
// summaries (onedev.kr FlashQLA talk summary, paragraph on parallelism).  One row block (FIX_ROWS rows
// of the state) per call, run by threads 0-255 of a CTA, which synchronise on named barrier 1.  The
// composition is serial over segments, but every step's inputs (M_j and E_j's rows) are independent of
// the chain, so they stream through a two-stage shared-memory ring, two bulk copies per step issued by
// one thread on the stage's mbarrier: step i computes while step i + 1's transition lands.  The segment start modes (which segments take the fix-up at all) are
// decided up front, one segment per thread.  Used by the stand-alone fix-up kernel and, as a work item
// of the single-launch sequence parallelism, by the tcgen05 recurrent kernels.
#pragma once
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

constexpr int FIX_MODES = 2048;  // segments per sequence whose modes are kept in shared memory

// The product cur M of a step: thread t takes the column pair t % (D/2) of all FIX_ROWS rows over one of
// the 512 / D parts of the k range, so that every element of M read from shared memory serves all
// FIX_ROWS rows; the parts' sums meet in shared memory.
static_assert(FIX_ROWS == 8, "the product reads a column of cur as two float4");
template <int D> __host__ __device__ constexpr int fix_kparts() { return 256 / (D / 2); }

// shared memory of one fix-up row block: the ring, cur (transposed: [k][row]), the partial sums, the
// working steps, the modes, the step count and the ring's two mbarriers
template <int D> constexpr size_t fixup_smem_bytes() {
  return 2 * ((size_t)D * D + FIX_ROWS * D) * sizeof(float) + FIX_ROWS * D * sizeof(float) +
         (size_t)fix_kparts<D>() * FIX_ROWS * D * sizeof(float) + FIX_MODES * 2 + FIX_MODES + 32;
}

__device__ __forceinline__ void fix_bar() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }

template <int D>
__device__ __forceinline__ void fixup_rows(const FixupArgs &a, int rb, int h, int n, unsigned char *smem) {
  using namespace umma;
  const int H = a.H;
  const int tid = threadIdx.x;
  const size_t DD = (size_t)D * D;
  float *ring = reinterpret_cast<float *>(smem);                  // 2 stages of [M (D x D) | E rows]
  constexpr int NKP = fix_kparts<D>();  // parts of the k range
  float *curT = ring + 2 * (DD + FIX_ROWS * D);  // [k][row]: the source segment's corrected rows
  float *red = curT + FIX_ROWS * D;             // [part][row][column] partial sums
  short *work = reinterpret_cast<short *>(red + NKP * FIX_ROWS * D);
  signed char *fix_mode = reinterpret_cast<signed char *>(work + FIX_MODES);
  int *nwork = reinterpret_cast<int *>(fix_mode + FIX_MODES);
  uint64_t *fbar = reinterpret_cast<uint64_t *>(fix_mode + FIX_MODES + 8);  // stage s lands on fbar[s]
  if (a.fixflag && *a.fixflag == 0) return;  // no segment of this direction needs the exact fix-up
  const int nseg = a.plan.seq_nseg[n];
  if (nseg <= 1) return;
  const int seg0 = a.plan.seq_seg0[n], chunk0 = a.plan.seq_chunk0[n];
  const int nchunks = (a.plan.seq_len[n] + CH - 1) / CH;
  const bool window = !(a.flags & kFlagWindowOff);
  constexpr int NCP = D / 2, KPP = D / NKP;  // column pairs; k per part
  const int cp = tid % NCP, kp = tid / NCP;   // product: columns 2 cp, 2 cp + 1, k in [kp KPP, kp KPP + KPP)
  constexpr int RPT = FIX_ROWS * D / 256;     // sums: rows fr0 .. fr0 + RPT - 1 of column fc
  const int fc = tid % D, fr0 = (tid / D) * RPT;
  // the start (end, reversed) mode of segment j
  auto start_mode = [&](int j) {
    int w;
    if (!a.reverse) return fwd_start_mode(a.gsum, H, h, chunk0, seg_begin(j, a.Lfirst, a.Lseg), j, window, &w);
    return bwd_start_mode(a.gsum, H, h, chunk0, min(seg_begin(j + 1, a.Lfirst, a.Lseg), nchunks), nchunks, j, nseg,
                          window, &w);
  };
  const bool small = nseg <= FIX_MODES;
  if (small) {
    for (int j = tid; j < nseg; j += 256) fix_mode[j] = start_mode(j) == START_FIXUP;
    fix_bar();
    if (tid == 0) {  // working steps in chain order: target jt, composed from js (forward js = jt - 1)
      int nw = 0;
      for (int step = 0; step < nseg - 1; ++step) {
        const int jt = a.reverse ? nseg - 2 - step : step + 1, js = a.reverse ? jt + 1 : jt - 1;
        if (fix_mode[jt]) work[nw++] = (short)(fix_mode[js] ? jt | 0x4000 : jt);
      }
      *nwork = nw;
    }
    fix_bar();
  }
  const int nw = small ? *nwork : nseg - 1;
  // step i -> (target jt, uses M); for very long plans the modes are evaluated on the fly
  auto step_of = [&](int i, int &jt, bool &withM) {
    if (small) {
      const int v = work[i];
      jt = v & 0x3fff;
      withM = (v & 0x4000) != 0;
      return true;
    }
    jt = a.reverse ? nseg - 2 - i : i + 1;
    if (start_mode(jt) != START_FIXUP) return false;
    withM = start_mode(a.reverse ? jt + 1 : jt - 1) == START_FIXUP;
    return true;
  };
  if (tid == 0) {
    mbar_init(smem_u32(&fbar[0]), 1);
    mbar_init(smem_u32(&fbar[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  fix_bar();
  // thread 0: step i's M (if used) and E rows into stage i & 1 by two bulk copies; a step with nothing to
  // load completes its stage's phase by a plain arrival
  auto issue = [&](int i) {
    if (tid != 0 || i >= nw) return;
    int jt;
    bool withM;
    const uint32_t bar = smem_u32(&fbar[i & 1]);
    if (step_of(i, jt, withM)) {
      const int js = a.reverse ? jt + 1 : jt - 1;
      const size_t src = ((size_t)(seg0 + js) * H + h) * DD;
      float *st = ring + (size_t)(i & 1) * (DD + FIX_ROWS * D);
      fence_async_smem();  // the stage's last generic reads (before the caller's barrier) precede the copies
      mbar_expect_tx(bar, (uint32_t)(((withM ? DD : 0) + FIX_ROWS * D) * sizeof(float)));
      if (withM) bulk_load(smem_u32(st), a.M + src, (uint32_t)(DD * sizeof(float)), bar);
      bulk_load(smem_u32(st + DD), a.E + src + (size_t)rb * FIX_ROWS * D, (uint32_t)(FIX_ROWS * D * sizeof(float)),
                bar);
    } else {
      mbar_arrive(bar);
    }
  };
  issue(0);
  issue(1);
  for (int i = 0; i < nw; ++i) {
    int jt;
    bool withM;
    const bool active = step_of(i, jt, withM);
    // step i's inputs have landed (step i + 1's may be in flight); an expired wait is recorded and the
    // composition goes on (its result is then not to be trusted)
    mbar_wait(smem_u32(&fbar[i & 1]), (i >> 1) & 1, a.status, 4);
    fix_bar();
    if (active) {
      const float *st = ring + (size_t)(i & 1) * (DD + FIX_ROWS * D);
      float v[RPT];  // E's rows, read before the barrier that lets the stage be refilled
#pragma unroll
      for (int t = 0; t < RPT; ++t) v[t] = st[DD + (fr0 + t) * D + fc];
      if (withM) {  // curT holds the corrected state of the source segment (the previous working step)
        float acc[FIX_ROWS][2] = {};
        const float *mk = st + (size_t)kp * KPP * D + 2 * cp;
        const float *xk = curT + kp * KPP * FIX_ROWS;
#pragma unroll 4
        for (int kk = 0; kk < KPP; ++kk) {
          const float2 m = *reinterpret_cast<const float2 *>(mk + (size_t)kk * D);
          const float4 x0 = *reinterpret_cast<const float4 *>(xk + kk * FIX_ROWS);
          const float4 x1 = *reinterpret_cast<const float4 *>(xk + kk * FIX_ROWS + 4);
          const float x[FIX_ROWS] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int r = 0; r < FIX_ROWS; ++r) {
            acc[r][0] = fmaf(x[r], m.x, acc[r][0]);
            acc[r][1] = fmaf(x[r], m.y, acc[r][1]);
          }
        }
#pragma unroll
        for (int r = 0; r < FIX_ROWS; ++r)
          *reinterpret_cast<float2 *>(red + (kp * FIX_ROWS + r) * D + 2 * cp) = make_float2(acc[r][0], acc[r][1]);
      }
      fix_bar();  // every thread has read curT and this stage; the partial sums are written
      if (withM) {
#pragma unroll
        for (int q = 0; q < NKP; ++q)
#pragma unroll
          for (int t = 0; t < RPT; ++t) v[t] += red[(q * FIX_ROWS + fr0 + t) * D + fc];
      }
      float *out = a.out + ((size_t)(seg0 + jt) * H + h) * DD + (size_t)(rb * FIX_ROWS + fr0) * D + fc;
#pragma unroll
      for (int t = 0; t < RPT; ++t) {
        curT[fc * FIX_ROWS + fr0 + t] = v[t];
        out[(size_t)t * D] = v[t];
      }
    } else {
      fix_bar();
    }
    issue(i + 2);  // into the stage just read
  }
  fix_bar();  // every wait on the ring's barriers is done (every issued step was awaited)
  if (tid == 0) {
    mbar_inval(smem_u32(&fbar[0]));
    mbar_inval(smem_u32(&fbar[1]));
  }
}

}  // namespace gdn
