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
#include "fixup.cuh"
#include "kernels.h"
#include "modes.cuh"

namespace gdn {

// One block.  Builds the per-sequence and per-segment tables; a malformed
// cu_seqlens (not starting at 0, decreasing, or not ending at T) sets status
// bit 1 and leaves every sequence empty, so the chunk kernels do nothing.
// Given the gate sums of a call whose forward computed them (modes != 0,
// gsum set), it also runs the fix-up mode scan over the tables it built.
__global__ void plan_kernel(Plan p, const int *cu, int N, int T, int Lseg, int Lfirst, int S_max, int CH_max, int *status,
                            int *zero, int nzero, const float *gsum, int H, int modes, unsigned flags, Sched fs,
                            Sched bs) {
  pdl_trigger();
  pdl_wait();
  __shared__ int carry_c, carry_s, bad;
  __shared__ int wsum_c[32], wsum_s[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid < 8 && status) status[tid] = 0;  // status word, fix-up flags, counters and tickets of this call
  for (int i = tid; i < nzero; i += nt) zero[i] = 0;  // the schedules' counters
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
    const int ns = (n < N && !isbad) ? seg_count(nc, Lfirst, Lseg) : 0;
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
    int2 ci = make_int2(0, 0);
    if (owner >= 0) {
      const int lc = c - p.seq_chunk0[owner];
      ci.x = p.seq_bos[owner] + lc * CH;
      ci.y = min(CH, p.seq_len[owner] - lc * CH);
    }
    p.chunk_info[c] = ci;
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
  if (!modes || !gsum) return;
  __syncthreads();  // the tables above, the zeroed status words and counters
  fixup_modes(p, gsum, H, Lseg, Lfirst, S_max, flags, status, tid, nt, fs, bs, N * H);
}

int launch_plan(const Plan &p, const int *cu, int N, int T, int Lseg, int Lfirst, int S_max, int CH_max, int *status,
                int *zero, int nzero, cudaStream_t st, const float *gsum, int H, int modes, unsigned flags,
                const Sched *sched) {
  Sched none;
  memset(&none, 0, sizeof none);
  return (int)launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, st, p, cu, N, T, Lseg, Lfirst, S_max, CH_max, status,
                         zero, zero ? nzero : 0, gsum, H, modes, flags, sched ? sched[0] : none, sched ? sched[1] : none);
}

// One block per global chunk: the chunk's log-gates of 32 heads at a time are
// staged in shared memory with coalesced row loads (tokens are rows of H gates),
// then one warp per head scans its 64 values: gsum[c, h] = sum of g over the
// chunk's tokens (each g raised to GATE_FLOOR first, as in the chunk kernels).
// With modes != 0 (a call with segments) the last block to finish also runs the fix-up mode scan
// over every (segment, head) (status[3] counts finished blocks; the plan kernel zeroed it).
__global__ void __launch_bounds__(256) gate_scan_kernel(Plan p, const float *g, int H, float *gsum, int *status,
                                                        int modes, int Lseg, int Lfirst, int S_max, unsigned flags,
                                                        Sched fs,
                                                        Sched bs, int NH) {
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
  fixup_modes(p, gsum, H, Lseg, Lfirst, S_max, flags, status, threadIdx.x, blockDim.x, fs, bs, NH);
}

int launch_gate_scan(const Plan &p, const float *g, int H, int CH_max, float *gsum, int *status, int modes, int Lseg,
                     int Lfirst, int S_max, unsigned flags, const Sched *sched, int NH, cudaStream_t st) {
  if (CH_max == 0) return 0;
  Sched none;
  memset(&none, 0, sizeof none);
  return (int)launch_pdl(gate_scan_kernel, dim3(CH_max), dim3(256), 0, st, p, g, H, gsum, status, modes, Lseg, Lfirst,
                         S_max, flags, sched ? sched[0] : none, sched ? sched[1] : none, NH);
}

// 256 threads; grid (D / FIX_ROWS, H, N), one fix-up row block per CTA (see fixup_rows), or, with a ticket
// counter, a 1-D grid whose CTAs take the row blocks in turn: a call whose segments need no fix-up (or
// few) then costs one short wave of CTAs instead of one CTA per row block
template <int D>
__global__ void __launch_bounds__(256, 1) fixup_kernel(FixupArgs a, int nitems) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char fx_smem[];
  if (!a.ticket) {
    fixup_rows<D>(a, blockIdx.x, blockIdx.y, blockIdx.z, fx_smem);
    return;
  }
  if (a.fixflag && *a.fixflag == 0) return;  // no segment of this direction needs the exact fix-up
  constexpr int NRB = D / FIX_ROWS;
  __shared__ int tk;
  for (;;) {
    if (threadIdx.x == 0) tk = atomicAdd(a.ticket, 1);
    __syncthreads();
    const int t = tk;
    __syncthreads();  // every thread has its ticket before thread 0 takes the next one
    if (t >= nitems) break;
    fixup_rows<D>(a, t % NRB, (t / NRB) % a.H, t / (NRB * a.H), fx_smem);
  }
}

int launch_fixup(const FixupArgs &a, int N, int ctas, cudaStream_t st) {
  if (N == 0) return 0;
  const int nitems = a.D / FIX_ROWS * a.H * N;
  const dim3 grid = (a.ticket && ctas > 0) ? dim3(min(ctas, nitems)) : dim3(a.D / FIX_ROWS, a.H, N);
  if (a.D == 128) {
    const size_t smem = fixup_smem_bytes<128>();
    cudaError_t e = cudaFuncSetAttribute(fixup_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)launch_pdl(fixup_kernel<128>, grid, dim3(256), smem, st, a, nitems);
  }
  if (a.D == 64) {
    const size_t smem = fixup_smem_bytes<64>();
    cudaError_t e = cudaFuncSetAttribute(fixup_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)launch_pdl(fixup_kernel<64>, grid, dim3(256), smem, st, a, nitems);
  }
  return -1;
}

}  // namespace gdn
