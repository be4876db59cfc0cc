// Segment plan, gate scan and the sequential start-state fix-up.
//
// Gate scan: "one light kernel scanning the gate distribution" decides which
// segment starts lie inside an effective sliding window (onedev.kr FlashQLA
// talk summary, paragraph on the effective sliding window).  Here it stores
// the log-decay sum of every (chunk, head); the chunk kernels derive from it
// the warm-up length of each segment start: the smallest w <= 8 chunks whose
// summed log-decay is <= ln(2^-24).  Because |I - beta k k^T|_2 <= 1 for unit
// keys and beta in [0, 1], starting w chunks early from a zero state leaves a
// start-state error below 2^-24 |S|, so that segment needs no correction.
//
// Fix-up: segments that are not inside a window get their exact start state
// from the composition S_start(j+1) = S_start(j) M_j + E_j over the segments of
// the sequence (onedev.kr talk summary, paragraph on parallelism).  Rows of the
// state are independent in this composition, so CTAs split the rows.
#include "kernels.h"

namespace gdn {

// One block.  Builds the per-sequence and per-segment tables; a malformed
// cu_seqlens (not starting at 0, decreasing, or not ending at T) sets status
// bit 1 and leaves every sequence empty, so the chunk kernels do nothing.
__global__ void plan_kernel(Plan p, const int *cu, int N, int T, int Lseg, int S_max, int CH_max, int *status) {
  pdl_trigger();
  pdl_wait();
  __shared__ int carry_c, carry_s, bad;
  __shared__ int wsum_c[32], wsum_s[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid < 4 && status) status[tid] = 0;  // status word and the fix-up flags of this call
  __syncthreads();
  if (tid == 0) {
    carry_c = 0;
    carry_s = 0;
    bad = 0;
    if (cu && (cu[0] != 0 || cu[N] != T)) bad = 1;
  }
  __syncthreads();
  if (cu) {
    for (int n = tid; n < N; n += nt)
      if (cu[n + 1] < cu[n]) atomicOr(&bad, 1);
  }
  __syncthreads();
  const bool isbad = bad != 0;
  if (isbad && tid == 0 && status) atomicOr(status, 2);
  for (int base = 0; base < N; base += nt) {
    const int n = base + tid;
    int len = 0, bos = 0;
    if (n < N && !isbad) {
      bos = cu ? cu[n] : n * T;
      len = cu ? cu[n + 1] - cu[n] : T;
    }
    const int nc = (len + CH - 1) / CH;
    // an empty sequence still gets one (chunk-less) segment: it passes S0 to S_T
    const int ns = (n < N && !isbad) ? max(1, (nc + Lseg - 1) / Lseg) : 0;
    // block-wide exclusive scans of nc and ns
    const int lane = tid & 31, warp = tid >> 5;
    int ic = nc, is = ns;
    for (int o = 1; o < 32; o <<= 1) {
      const int yc = __shfl_up_sync(0xffffffffu, ic, o), ys = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) {
        ic += yc;
        is += ys;
      }
    }
    if (lane == 31) {
      wsum_c[warp] = ic;
      wsum_s[warp] = is;
    }
    __syncthreads();
    if (warp == 0) {
      const int nw = nt / 32;
      int vc = lane < nw ? wsum_c[lane] : 0, vs = lane < nw ? wsum_s[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xffffffffu, vc, o), ys = __shfl_up_sync(0xffffffffu, vs, o);
        if (lane >= o) {
          vc += yc;
          vs += ys;
        }
      }
      if (lane < nw) {
        wsum_c[lane] = vc;
        wsum_s[lane] = vs;
      }
    }
    __syncthreads();
    const int pre_c = carry_c + (warp ? wsum_c[warp - 1] : 0) + ic - nc;
    const int pre_s = carry_s + (warp ? wsum_s[warp - 1] : 0) + is - ns;
    if (n < N) {
      p.seq_bos[n] = bos;
      p.seq_len[n] = len;
      p.seq_chunk0[n] = pre_c;
      p.seq_seg0[n] = pre_s;
      p.seq_nseg[n] = ns;
    }
    __syncthreads();
    if (tid == nt - 1) {
      carry_c = pre_c + nc;
      carry_s = pre_s + ns;
    }
    __syncthreads();
  }
  const int tot_c = carry_c, tot_s = carry_s;
  if (tid == 0) {
    p.totals[0] = tot_c;
    p.totals[1] = tot_s;
    if ((tot_c > CH_max || tot_s > S_max) && status) atomicOr(status, 2);
  }
  // owner sequence of every chunk and segment: the last sequence whose prefix is
  // <= the index (an empty sequence shares its prefix with the next one, so the
  // search never lands on it for an index below the total)
  for (int c = tid; c < CH_max; c += nt) {
    int owner = -1;
    if (c < tot_c && tot_c <= CH_max) {
      int lo = 0, hi = N - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seq_chunk0[mid] <= c) lo = mid; else hi = mid - 1;
      }
      owner = lo;
    }
    p.chunk_seq[c] = owner;
  }
  for (int s = tid; s < S_max; s += nt) {
    int owner = -1;
    if (s < tot_s && tot_s <= S_max) {
      int lo = 0, hi = N - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seq_seg0[mid] <= s) lo = mid; else hi = mid - 1;
      }
      owner = lo;
    }
    p.seg_seq[s] = owner;
  }
}

int launch_plan(const Plan &p, const int *cu, int N, int T, int Lseg, int S_max, int CH_max, int *status,
                cudaStream_t st) {
  return (int)launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, st, p, cu, N, T, Lseg, S_max, CH_max, status);
}

// One block per global chunk: the chunk's log-gates of 32 heads at a time are
// staged in shared memory with coalesced row loads (tokens are rows of H gates),
// then one warp per head scans its 64 values: gsum[c, h] = sum of g over the
// chunk's tokens (each g raised to GATE_FLOOR first, as in the chunk kernels).
__device__ void fixup_modes(const Plan &p, const float *gsum, int H, int Lseg, int S_max, unsigned flags, int *status,
                            int i0, int stride);

// With modes != 0 (a call with segments) the last block to finish also runs the fix-up mode scan
// over every (segment, head) (status[3] counts finished blocks; the plan kernel zeroed it).
__global__ void __launch_bounds__(256) gate_scan_kernel(Plan p, const float *g, int H, float *gsum, int *status,
                                                        int modes, int Lseg, int S_max, unsigned flags) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[CH][33];
  __shared__ int last;
  const int c = blockIdx.x;
  const int n = p.chunk_seq[c];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (n < 0) {
    for (int h = threadIdx.x; h < H; h += blockDim.x) gsum[(size_t)c * H + h] = 0.f;
  } else {
  const int lc = c - p.seq_chunk0[n];
  const long tok0 = (long)p.seq_bos[n] + (long)lc * CH;
  const int nvalid = min(CH, p.seq_len[n] - lc * CH);
  for (int h0 = 0; h0 < H; h0 += 32) {
    const int hh = h0 + lane;
    for (int r = warp; r < CH; r += 8) tile[r][lane] = (r < nvalid && hh < H) ? g[(size_t)(tok0 + r) * H + hh] : 0.f;
    __syncthreads();
    for (int hl = warp; hl < 32 && h0 + hl < H; hl += 8) {
      float a = fmaxf(tile[lane][hl], GATE_FLOOR), b = fmaxf(tile[lane + 32][hl], GATE_FLOOR);
      for (int o = 1; o < 32; o <<= 1) {
        const float ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) {
          a += ya;
          b += yb;
        }
      }
      const float Gmid = __shfl_sync(0xffffffffu, a, 31);
      b += Gmid;
      const float Glast = __shfl_sync(0xffffffffu, b, 31);
      if (lane == 0) gsum[(size_t)c * H + h0 + hl] = Glast;
    }
    __syncthreads();
  }
  }
  if (!modes) return;
  // last block: every block's gsum writes are visible once it has fenced and counted itself
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(status + 3, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  fixup_modes(p, gsum, H, Lseg, S_max, flags, status, threadIdx.x, blockDim.x);
}

int launch_gate_scan(const Plan &p, const float *g, int H, int CH_max, float *gsum, int *status, int modes, int Lseg,
                     int S_max, unsigned flags, cudaStream_t st) {
  if (CH_max == 0) return 0;
  return (int)launch_pdl(gate_scan_kernel, dim3(CH_max), dim3(256), 0, st, p, g, H, gsum, status, modes, Lseg, S_max,
                         flags);
}

// Does any segment start (forward) or end (reverse) need the exact fix-up?  status[1] / status[2]
// become nonzero if so; the pass-A launches and the fix-ups of a direction without any such segment
// return at once.  (segment, head) pairs i0, i0 + stride, ...; gsum read through L2 (other blocks
// wrote it in this launch).
__device__ void fixup_modes(const Plan &p, const float *gsum, int H, int Lseg, int S_max, unsigned flags, int *status,
                            int i0, int stride) {
  const bool window = !(flags & kFlagWindowOff);
  bool fwd_fix = false, bwd_fix = false;
  for (int i = i0; i < S_max * H; i += stride) {
    const int s = i / H, h = i % H;
    const int n = __ldcg(p.seg_seq + s);
    if (n < 0) continue;
    const int j = s - __ldcg(p.seq_seg0 + n), nseg = __ldcg(p.seq_nseg + n), chunk0 = __ldcg(p.seq_chunk0 + n);
    const int nchunks = (__ldcg(p.seq_len + n) + CH - 1) / CH;
    const int cbeg = j * Lseg, cend = min((j + 1) * Lseg, nchunks);
    // the start-mode rules of the chunk kernels, on L2-coherent loads of gsum: all WMAX sums of
    // each window are loaded at once (no dependent load chain), then scanned
    if (j > 0) {
      float gs[WMAX];
#pragma unroll
      for (int ww = 1; ww <= WMAX; ++ww) gs[ww - 1] = ww <= cbeg ? __ldcg(gsum + (size_t)(chunk0 + cbeg - ww) * H + h) : 0.f;
      bool warm = false;
      if (window) {
        float acc = 0.f;
#pragma unroll
        for (int ww = 1; ww <= WMAX; ++ww) {
          acc += gs[ww - 1];
          warm |= ww <= cbeg && acc <= LN_EPS_WINDOW;
        }
      }
      fwd_fix |= !warm;
    }
    if (j < nseg - 1) {
      float gs[WMAX];
#pragma unroll
      for (int ww = 1; ww <= WMAX; ++ww)
        gs[ww - 1] = cend + ww <= nchunks ? __ldcg(gsum + (size_t)(chunk0 + cend + ww - 1) * H + h) : 0.f;
      bool warm = false;
      if (window) {
        float acc = 0.f;
#pragma unroll
        for (int ww = 1; ww <= WMAX; ++ww) {
          acc += gs[ww - 1];
          warm |= cend + ww <= nchunks && acc <= LN_EPS_WINDOW;
        }
      }
      bwd_fix |= !warm;
    }
  }
  if (fwd_fix) atomicOr(status + 1, 1);
  if (bwd_fix) atomicOr(status + 2, 1);
}

// Start-state fix-up (forward: S_start[j+1] = S_start[j] M_j + E_j over the segments of one (sequence,
// head); the reverse chain mirrors it), the sequential composition of the segment summaries
// (onedev.kr talk summary, paragraph on parallelism).  grid (D / FIX_ROWS, H, N): FIX_ROWS rows of the
// state per CTA, 256 threads.  The composition is serial over segments, but every step's inputs (M_j
// and E_j's rows) are independent of the chain, so they stream through a two-stage shared-memory ring
// by cp.async: step i computes while step i + 1's 64 KB transition lands.  The segment start modes
// (which segments take the fix-up at all) are decided up front, one segment per thread.
constexpr int FIX_ROWS = 8;
constexpr int FIX_MODES = 2048;  // segments per sequence whose modes are kept in shared memory

template <int D> constexpr size_t fixup_smem_bytes() { return 2 * ((size_t)D * D + FIX_ROWS * D) * sizeof(float); }

template <int D>
__global__ void __launch_bounds__(256, 1) fixup_kernel(FixupArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) float fx_sm[];  // 2 stages of [M (D x D) | E rows (FIX_ROWS x D)]
  __shared__ float cur[FIX_ROWS][D];
  __shared__ signed char fix_mode[FIX_MODES];  // per segment: 0 no fix-up, 1 fix-up from E alone, 2 from E and M
  __shared__ int nwork;
  __shared__ short work[FIX_MODES];            // target segment of each working step, in chain order
  const int rb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = a.H;
  if (a.fixflag && *a.fixflag == 0) return;  // no segment of this direction needs the exact fix-up
  const int nseg = a.plan.seq_nseg[n];
  if (nseg <= 1) return;
  const int seg0 = a.plan.seq_seg0[n], chunk0 = a.plan.seq_chunk0[n];
  const int nchunks = (a.plan.seq_len[n] + CH - 1) / CH;
  const bool window = !(a.flags & kFlagWindowOff);
  const size_t DD = (size_t)D * D;
  constexpr int CPT = D / 32;  // columns per thread
  const int tid = threadIdx.x;
  const int r = tid >> 5;
  const int c0 = (tid & 31) * CPT;
  const int row = rb * FIX_ROWS + r;
  // mode of segment j as the target of a fix-up step: is its start (end, reversed) corrected, and is the
  // segment it is composed from itself corrected (then its transition M takes part)
  auto start_mode = [&](int j) {
    int w;
    if (!a.reverse) return fwd_start_mode(a.gsum, H, h, chunk0, j * a.Lseg, j, window, &w);
    return bwd_start_mode(a.gsum, H, h, chunk0, min((j + 1) * a.Lseg, nchunks), nchunks, j, nseg, window, &w);
  };
  const bool small = nseg <= FIX_MODES;
  if (small) {
    for (int j = tid; j < nseg; j += blockDim.x) fix_mode[j] = start_mode(j) == START_FIXUP;
    __syncthreads();
    if (tid == 0) {  // working steps in chain order: target jt, composed from js (forward js = jt - 1)
      int nw = 0;
      for (int step = 0; step < nseg - 1; ++step) {
        const int jt = a.reverse ? nseg - 2 - step : step + 1, js = a.reverse ? jt + 1 : jt - 1;
        if (fix_mode[jt]) work[nw++] = (short)(fix_mode[js] ? jt | 0x4000 : jt);
      }
      nwork = nw;
    }
    __syncthreads();
  }
  const int nw = small ? nwork : nseg - 1;
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
  auto issue = [&](int i) {  // cp.async of step i's M (if used) and E rows into stage i & 1
    int jt;
    bool withM;
    if (i < nw && step_of(i, jt, withM)) {
      const int js = a.reverse ? jt + 1 : jt - 1;
      const size_t src = ((size_t)(seg0 + js) * H + h) * DD;
      float *st = fx_sm + (size_t)(i & 1) * (DD + FIX_ROWS * D);
      if (withM)
        for (int e = tid; e < (int)(DD / 4); e += blockDim.x) cp_async16(st + 4 * e, a.M + src + 4 * e, true);
      for (int e = tid; e < FIX_ROWS * D / 4; e += blockDim.x)
        cp_async16(st + DD + 4 * e, a.E + src + (size_t)rb * FIX_ROWS * D + 4 * e, true);
    }
    cp_async_commit();  // one group per step, empty or not
  };
  issue(0);
  issue(1);
  for (int i = 0; i < nw; ++i) {
    int jt;
    bool withM;
    const bool active = step_of(i, jt, withM);
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // step i's group has landed (i + 1's may be in flight)
    __syncthreads();
    if (active) {
      const float *st = fx_sm + (size_t)(i & 1) * (DD + FIX_ROWS * D);
      float acc[CPT];
#pragma unroll
      for (int t = 0; t < CPT; ++t) acc[t] = st[DD + r * D + c0 + t];
      if (withM) {  // cur holds the corrected state of the source segment (the previous working step)
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
          const float x = cur[r][k];
          float m[CPT];
          if constexpr (CPT == 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(st + (size_t)k * D + c0);
            m[0] = t4.x;
            m[1] = t4.y;
            m[2] = t4.z;
            m[3] = t4.w;
          } else {
            const float2 t2 = *reinterpret_cast<const float2 *>(st + (size_t)k * D + c0);
            m[0] = t2.x;
            m[1] = t2.y;
          }
#pragma unroll
          for (int t = 0; t < CPT; ++t) acc[t] = fmaf(x, m[t], acc[t]);
        }
      }
      __syncthreads();  // every thread has read cur and this stage
      float *out = a.out + ((size_t)(seg0 + jt) * H + h) * DD + (size_t)row * D;
#pragma unroll
      for (int t = 0; t < CPT; ++t) {
        cur[r][c0 + t] = acc[t];
        out[c0 + t] = acc[t];
      }
    } else {
      __syncthreads();
    }
    issue(i + 2);  // into the stage just read
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

int launch_fixup(const FixupArgs &a, int N, cudaStream_t st) {
  if (N == 0) return 0;
  dim3 grid(a.D / FIX_ROWS, a.H, N);
  if (a.D == 128) {
    const size_t smem = fixup_smem_bytes<128>();
    cudaError_t e = cudaFuncSetAttribute(fixup_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)launch_pdl(fixup_kernel<128>, grid, dim3(256), smem, st, a);
  }
  if (a.D == 64) {
    const size_t smem = fixup_smem_bytes<64>();
    cudaError_t e = cudaFuncSetAttribute(fixup_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)launch_pdl(fixup_kernel<64>, grid, dim3(256), smem, st, a);
  }
  return -1;
}

}  // namespace gdn
