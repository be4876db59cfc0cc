// C ABI of the library: argument validation, workspace layout, segment-length
// choice and the launch sequence of the forward and backward passes.
#include <algorithm>
#include <array>
#include <cmath>
#include <functional>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gdn.h"
#include "kernels.h"

using namespace gdn;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int num_sms() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    cache[dev] = v;
  }
  return cache[dev];
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  int N = 0, H = 0, D = 0, Tseq = 0;  // Tseq: per-sequence length for uniform batches, 0 for packed
  long Ttot = 0;
  int CH_max = 0, S_max = 0, Lseg = 1, Lfirst = 1;  // segment lengths in chunks: the first, then Lseg each
  bool sp = false;  // more than one segment possible for some sequence
  size_t esize = 2;
  size_t off_status = 0, off_plan = 0, off_gsum = 0;
  size_t off_sched = 0, off_lists = 0;  // single-launch sequence parallelism: zeroed counters, work lists
  int sched_zero = 0;                   // ints of the zeroed counter region
  size_t off_E = 0, off_M = 0, off_S = 0;     // forward fix-up buffers
  size_t off_states = 0, off_dstates = 0;   // backward per-chunk states
  size_t off_F = 0, off_R = 0, off_dS = 0;  // reverse fix-up buffers
  size_t off_dut = 0, dut_bytes = 0;        // the chain's per-chunk dUt^T and fp16 dO tiles (bf16, d = 128)
  size_t off_t64 = 0, off_t128 = 0;        // recomputed chunk context tiles (bf16, d = 128)
  size_t t64_bytes = 0, t128_bytes = 0;
  size_t off_tqkv = 0, off_nrm = 0, tqkv_bytes = 0, nrm_bytes = 0;
  size_t states_bytes = 0;                  // per-chunk start states
  size_t bwd_saved_total = 0;               // backward workspace when the forward saved its context
  size_t saved_off_t64 = 0, saved_off_t128 = 0, saved_off_tqkv = 0, saved_off_nrm = 0, saved_off_gsum = 0;
  size_t saved_total = 0;  // saved context: [states][t64][t128][tqkv][nrm][gsum]
  size_t off_fctx_t64 = 0, off_fctx_tqkv = 0;  // the plain forward's chunk context (bf16, d = 128)
  size_t fwd_core = 0, fwd_total = 0, bwd_total = 0;
};

// Does a plan of S segments per sequence over nh equal-length (sequence, head) pairs run the recurrent
// passes on the balanced grid (later segments one CTA each, the first segments sharing the other SMs)?
bool balanced_plan(long nh, int S, long slots) { return S >= 2 && nh * S > slots && nh * (S - 1) < slots; }

// Modelled time of the two recurrent passes (the forward's state pass and the backward's reverse
// chain) for a first segment of F chunks and later ones of L.  One CTA per (segment, head) walks its
// chunks serially and holds a whole SM; the hardware starts the CTAs in launch order (segments of a
// head, heads in turn) on whichever SM frees first, so the pass takes the makespan of that list on the
// SMs.  A segment costs a fixed part plus its chunks, plus kWarmChunks warm-up chunks where it does not
// start (forward) or end (reverse) its sequence (the window case of the gate scan; the exact case adds a
// pass A that the host cannot foresee, since it depends on the gates).  On the balanced grid the pass
// takes the longer of a later segment and the first segments of the most loaded shared CTA, each of
// which pays the fixed part of an item that follows another in the same CTA.  The constants fit GB300
// timings of the tcgen05 kernels (bench.py --sweep-seg-chunks over 21 plans of the H = 32, T = 8192
// prefill and 12 of the B = 4, H = 16, T = 4096 batch: one segment length 8 .. 128 chunks and first
// segments of 2 .. 20 chunks); the d = 64 and fp32 kernels are costed the same way.  Packed batches,
// whose lengths the host does not see, are costed in whole waves of an average item.
struct PassCost {
  double item_us, chunk_us, next_item_us;  // next_item_us: an item after another one in the same CTA
};
constexpr PassCost kFwdPass = {20.0, 3.2, 24.0}, kChainPass = {12.0, 2.9, 17.0};
constexpr int kWarmChunks = 2;

bool tc_shape(const gdn_shape &s) { return s.dtype == GDN_BF16 && s.Dk == 128; }

void plan_cost_us(const gdn_shape &s, int N, int maxc, int CH_max, int L, int F, double *fwd_us, double *bwd_us) {
  const int slots = num_sms();
  L = std::max(1, std::min(L, maxc));
  F = std::max(1, std::min(F, maxc));
  const int S = seg_count(maxc, F, L);
  const long nh = (long)N * s.H;
  const long items = s.cu_seqlens ? (long)std::ceil(s.H * ((double)CH_max / L + 0.5 * N)) : nh * S;
  if (s.cu_seqlens || items > 16L * slots) {
    const double waves = std::ceil((double)items / slots);
    const double steps = L + (L < maxc ? kWarmChunks : 0);
    *fwd_us = waves * (kFwdPass.item_us + steps * kFwdPass.chunk_us);
    *bwd_us = waves * (kChainPass.item_us + steps * kChainPass.chunk_us);
    return;
  }
  // chunk steps of segment j, its warm-up included
  auto seg_len = [&](int j) { return std::min(seg_begin(j + 1, F, L), maxc) - seg_begin(j, F, L); };
  auto steps = [&](int pass, int j) {
    if (pass == 0) return seg_len(j) + (j ? std::min(kWarmChunks, seg_begin(j, F, L)) : 0);
    const int cend = std::min(seg_begin(j + 1, F, L), maxc);
    return seg_len(j) + (j < S - 1 ? std::min(kWarmChunks, maxc - cend) : 0);
  };
  double out[2];
  if (tc_shape(s) && balanced_plan(nh, S, slots)) {
    const long shared = slots - nh * (S - 1), per_cta = (nh + shared - 1) / shared;
    for (int pass = 0; pass < 2; ++pass) {
      const PassCost &pc = pass ? kChainPass : kFwdPass;
      double big = 0.0;
      for (int j = 1; j < S; ++j) big = std::max(big, pc.item_us + steps(pass, j) * pc.chunk_us);
      out[pass] = std::max(big, per_cta * (pc.next_item_us + steps(pass, 0) * pc.chunk_us));
    }
  } else {
    for (int pass = 0; pass < 2; ++pass) {
      const PassCost &pc = pass ? kChainPass : kFwdPass;
      std::vector<double> sm(std::min<long>(slots, items), 0.0);  // a min-heap of the SMs' free times
      for (long i = 0; i < items; ++i) {
        const int j = (int)(i % S);  // launch order: the segments of one (sequence, head), then the next
        const double d = pc.item_us + steps(pass, j) * pc.chunk_us;
        if ((long)i < (long)sm.size()) {
          sm[i] = d;
          std::push_heap(sm.begin(), sm.begin() + i + 1, std::greater<double>());
        } else {
          std::pop_heap(sm.begin(), sm.end(), std::greater<double>());
          sm.back() += d;
          std::push_heap(sm.begin(), sm.end(), std::greater<double>());
        }
      }
      out[pass] = *std::max_element(sm.begin(), sm.end());
    }
  }
  *fwd_us = out[0];
  *bwd_us = out[1];
}

// Segment lengths: L chunks per segment after a first segment of F.  With few (sequence, head) pairs the
// sequences are split until the work items fill the SMs (onedev.kr FlashQLA talk summary, paragraph on
// parallelism: one head per SM leaves most of a >100-SM card idle); the plan minimises the modelled time
// of the two recurrent passes over the lengths that give each segment count its shortest longest segment,
// up to 16 waves of items, and, for the tcgen05 kernels on equal-length sequences, over the balanced plans
// (a shorter first segment of at least min(WMAX, L) chunks, so that the next segment's warm-up is never cut
// short by it).  Results are cached per shape class (the plan is chosen on every call).
void choose_plan(const gdn_shape &s, int N, int maxc, int CH_max, int &L, int &F) {
  L = F = std::max(1, maxc);
  if (maxc <= 0) return;
  if (s.flags & GDN_SP_OFF) return;
  if (s.seg_chunks > 0) {
    L = s.seg_chunks;
    F = s.seg_first > 0 ? s.seg_first : L;
    return;
  }
  const int slots = num_sms();
  const long nh = (long)N * s.H;
  if (nh >= slots) return;
  static std::mutex mu;
  static std::vector<std::array<long, 7>> cache;  // {N, H, maxc, CH_max, packed, SMs, tcgen05}
  static std::vector<std::pair<int, int>> cached;
  const std::array<long, 7> key = {N, s.H, maxc, CH_max, s.cu_seqlens != nullptr, slots, tc_shape(s)};
  {
    std::lock_guard<std::mutex> lk(mu);
    for (size_t i = 0; i < cache.size(); ++i)
      if (cache[i] == key) {
        L = cached[i].first;
        F = cached[i].second;
        return;
      }
  }
  int bestL = maxc, bestF = maxc;
  double best_cost = 1e300;
  auto consider = [&](int l, int f) {
    double fw, bw;
    plan_cost_us(s, N, maxc, CH_max, l, f, &fw, &bw);
    if (fw + bw < best_cost - 1e-9) {
      best_cost = fw + bw;
      bestL = l;
      bestF = f;
    }
  };
  int prevL = 0;
  for (int S = 1; S <= maxc; ++S) {
    const int l = (maxc + S - 1) / S;
    if (l == prevL) continue;
    prevL = l;
    if (nh * S > 16L * slots) break;
    consider(l, l);
  }
  if (!s.cu_seqlens && tc_shape(s)) {
    for (int S = 2; S <= maxc && nh * (S - 1) < slots; ++S) {
      if (!balanced_plan(nh, S, slots)) continue;
      for (int f = 1; f < maxc; ++f) {
        const int l = (maxc - f + S - 2) / (S - 1);
        if (l < 1 || f < std::min(WMAX, l) || seg_count(maxc, f, l) != S) continue;
        consider(l, f);
      }
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() > 256) {
    cache.clear();
    cached.clear();
  }
  cache.push_back(key);
  cached.push_back({bestL, bestF});
  L = bestL;
  F = bestF;
}

int make_layout(const gdn_shape *s, Layout &L) {
  if (!s) return fail(GDN_ERR_INVALID_ARG, "shape is NULL");
  if (s->reserved[0] || s->reserved[1]) return fail(GDN_ERR_INVALID_ARG, "reserved fields must be 0");
  if (s->B < 1 || s->T < 0 || s->H < 1) return fail(GDN_ERR_INVALID_ARG, "need B >= 1, T >= 0, H >= 1");
  if (s->Dk != s->Dv) return fail(GDN_ERR_UNSUPPORTED, "d_k != d_v is not supported");
  if (s->Dk != 64 && s->Dk != 128) return fail(GDN_ERR_UNSUPPORTED, "d must be 64 or 128 (got %d)", s->Dk);
  if (s->dtype != GDN_BF16 && s->dtype != GDN_FP32) return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
  if (s->dtype == GDN_FP32 && s->Dk != 64) return fail(GDN_ERR_UNSUPPORTED, "fp32 mode supports d = 64 only");
  if (s->seg_chunks < 0) return fail(GDN_ERR_INVALID_ARG, "seg_chunks must be >= 0");
  if (s->seg_first < 0) return fail(GDN_ERR_INVALID_ARG, "seg_first must be >= 0");
  if (s->seg_first > 0 && s->seg_chunks == 0) return fail(GDN_ERR_INVALID_ARG, "seg_first needs seg_chunks > 0");
  if (!std::isfinite(s->scale) || s->scale == 0.f) return fail(GDN_ERR_INVALID_ARG, "scale must be finite and non-zero");
  if (s->cu_seqlens) {
    if (s->B != 1) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens requires B == 1");
    if (s->num_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens requires num_seqs >= 1");
    L.N = s->num_seqs;
    L.Tseq = 0;
  } else {
    L.N = s->B;
    L.Tseq = s->T;
  }
  if ((long)s->B * s->T > (long)INT32_MAX / 2) return fail(GDN_ERR_UNSUPPORTED, "too many tokens");
  L.H = s->H;
  L.D = s->Dk;
  L.Ttot = (long)s->B * s->T;
  L.esize = s->dtype == GDN_BF16 ? 2 : 4;
  int maxc;
  if (s->cu_seqlens) {
    L.CH_max = (int)((L.Ttot + (long)(CH - 1) * L.N) / CH);
    maxc = (int)((L.Ttot + CH - 1) / CH);
  } else {
    maxc = (s->T + CH - 1) / CH;
    L.CH_max = L.N * maxc;
  }
  // the context tiles of the tcgen05 path are addressed by 32-bit TMA row coordinates (the largest map,
  // the five 64-row tiles per (chunk, head), has CH_max * H * 320 rows)
  if (s->dtype == GDN_BF16 && L.D == 128 && (long)L.CH_max * L.H * T64_TILES * CH > (long)INT32_MAX)
    return fail(GDN_ERR_UNSUPPORTED, "too many (chunk, head) pairs for the context tiles (%ld, at most %ld)",
                (long)L.CH_max * L.H, (long)INT32_MAX / (T64_TILES * CH));
  choose_plan(*s, L.N, maxc, L.CH_max, L.Lseg, L.Lfirst);
  // a sequence of nc chunks has at most 2 + nc / Lseg segments
  if (s->cu_seqlens) L.S_max = L.CH_max / L.Lseg + 2 * L.N + 1;
  else L.S_max = L.N * seg_count(maxc, L.Lfirst, L.Lseg);
  L.sp = std::min(L.Lfirst, L.Lseg) < maxc;
  const size_t DD = (size_t)L.D * L.D;
  const size_t nplan = 5 * (size_t)L.N + L.S_max + 3 * (size_t)L.CH_max + 2;
  size_t off = 0;
  L.off_status = off;
  off += 256;
  L.off_plan = off;
  off = align256(off + nplan * 4);
  L.off_gsum = off;
  off = align256(off + (size_t)L.CH_max * L.H * 4);
  // the two directions' schedules: [hdr fwd | hdr bwd | needA, doneA, doneF fwd | the same bwd] (zeroed by the
  // plan kernel), then per direction listA [2 S_max H], listBn, listBf [S_max H], listF [N H]
  L.off_sched = off;
  L.sched_zero = L.sp ? 2 * SCHED_HDR + 6 * L.N * L.H : 0;
  off = align256(off + (size_t)L.sched_zero * 4);
  L.off_lists = off;
  if (L.sp) off = align256(off + (size_t)2 * (4 * (size_t)L.S_max * L.H + (size_t)L.N * L.H) * 4);
  const size_t spbuf = L.sp ? align256((size_t)L.S_max * L.H * DD * 4) : 0;
  L.off_E = off;
  off += spbuf;
  L.off_M = off;
  off += spbuf;
  L.off_S = off;
  off += spbuf;
  L.fwd_core = off;
  const bool tiles = s->dtype == GDN_BF16 && L.D == 128;
  L.t64_bytes = tiles ? align256((size_t)L.CH_max * L.H * T64_TILES * CH * CH * 2) : 0;
  L.t128_bytes = tiles ? align256((size_t)L.CH_max * L.H * T128_TILES * 128 * CH * 2) : 0;
  L.tqkv_bytes = tiles ? align256((size_t)L.CH_max * L.H * TQ_TILES * CH * 128 * 2) : 0;
  L.nrm_bytes = tiles ? align256((size_t)L.CH_max * L.H * 2 * CH * 4) : 0;
  // a forward that saves no context still passes the chunk-local half's tiles to the recurrent half
  L.off_fctx_t64 = off;
  off += L.t64_bytes;
  L.off_fctx_tqkv = off;
  off += L.tqkv_bytes;
  L.fwd_total = off;
  // backward (its own call: it reuses the forward-only context region): the reverse-chain buffers
  // first, then the per-chunk states and context tiles that the backward recomputes unless the
  // forward saved them (a saved-context backward needs only the prefix up to bwd_saved_total)
  off = L.fwd_core;
  L.states_bytes = align256((size_t)L.CH_max * L.H * DD * L.esize);
  L.off_dstates = off;
  off += L.states_bytes;
  L.off_F = off;
  off += spbuf;
  L.off_R = off;
  off += spbuf;
  L.off_dS = off;
  off += spbuf;
  L.dut_bytes = tiles ? align256((size_t)L.CH_max * L.H * TC_TILES * 128 * CH * 2) : 0;
  L.off_dut = off;
  off += L.dut_bytes;
  L.bwd_saved_total = off;
  L.off_states = off;
  off += L.states_bytes;
  L.off_t64 = off;
  off += L.t64_bytes;
  L.off_t128 = off;
  off += L.t128_bytes;
  L.off_tqkv = off;
  off += L.tqkv_bytes;
  L.off_nrm = off;
  off += L.nrm_bytes;
  L.bwd_total = off;
  L.saved_off_t64 = L.states_bytes;
  L.saved_off_t128 = L.states_bytes + L.t64_bytes;
  L.saved_off_tqkv = L.saved_off_t128 + L.t128_bytes;
  L.saved_off_nrm = L.saved_off_tqkv + L.tqkv_bytes;
  // the per-(chunk, head) gate sums: the saved-context backward takes them instead of rescanning g
  L.saved_off_gsum = L.saved_off_nrm + L.nrm_bytes;
  L.saved_total = L.saved_off_gsum + align256((size_t)L.CH_max * L.H * 4);
  return GDN_OK;
}

// The work lists of one direction (0 forward, 1 reverse) of the single-launch sequence parallelism.
Sched sched_of(const Layout &L, char *ws, int dir) {
  int *z = reinterpret_cast<int *>(ws + L.off_sched);
  int *lists = reinterpret_cast<int *>(ws + L.off_lists);
  const size_t NH = (size_t)L.N * L.H, SH = (size_t)L.S_max * L.H;
  Sched sc;
  sc.hdr = z + dir * SCHED_HDR;
  sc.needA = z + 2 * SCHED_HDR + dir * 3 * NH;
  sc.doneA = sc.needA + NH;
  sc.doneF = sc.doneA + NH;
  sc.listA = lists + dir * (4 * SH + NH);
  sc.listBn = sc.listA + 2 * SH;
  sc.listBf = sc.listBn + SH;
  sc.listF = sc.listBf + SH;
  return sc;
}

// Is sequence parallelism run as one launch per direction?  On request (GDN_SP_SINGLE_LAUNCH), for the tcgen05
// path (bf16, d = 128) with segments.
bool single_launch_sp(const Layout &L, const gdn_shape *s) {
  return (s->flags & GDN_SP_SINGLE_LAUNCH) && L.sp && s->dtype == GDN_BF16 && L.D == 128 && L.Ttot > 0;
}
// CTAs of such a launch: one per possible work item (pass A two roles, pass B, fix-up row blocks)
unsigned sched_grid(const Layout &L) {
  return (unsigned)(3 * L.S_max * L.H + (L.D / FIX_ROWS) * L.N * L.H);
}

Plan plan_of(const Layout &L, char *ws) {
  Plan pl;
  pl.chunk_info = reinterpret_cast<int2 *>(ws + L.off_plan);
  int *p = reinterpret_cast<int *>(pl.chunk_info + L.CH_max);
  pl.seq_bos = p;
  pl.seq_len = p + L.N;
  pl.seq_chunk0 = p + 2 * L.N;
  pl.seq_seg0 = p + 3 * L.N;
  pl.seq_nseg = p + 4 * L.N;
  pl.seg_seq = p + 5 * L.N;
  pl.chunk_seq = pl.seg_seq + L.S_max;
  pl.totals = pl.chunk_seq + L.CH_max;
  return pl;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_ptrs(std::initializer_list<std::pair<const void *, const char *>> req,
               std::initializer_list<std::pair<const void *, const char *>> opt) {
  for (auto &x : req) {
    if (!x.first) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", x.second);
    if (!aligned16(x.first)) return fail(GDN_ERR_INVALID_ARG, "%s is not 16-byte aligned", x.second);
  }
  for (auto &x : opt)
    if (x.first && !aligned16(x.first)) return fail(GDN_ERR_INVALID_ARG, "%s is not 16-byte aligned", x.second);
  return GDN_OK;
}

// ------------------------------------------------------------------ profiler
// Optional per-launch CUDA-event timing (diagnostics for benchmarks): when
// enabled, every kernel launch is bracketed by two events from a fixed pool on
// the launch stream; gdn_profile_report() sums the durations per kernel name.
struct ProfRec {
  const char *name;
  int ev0, ev1;
};
struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool;
  int used = 0;
  std::vector<ProfRec> recs;
  std::vector<std::string> names;
  std::vector<double> total_ms;
  std::vector<long> count;
  std::string only;  // bracket only launches of this name ("" = every launch)
};
Profiler g_prof;

struct ProfScope {
  int idx = -1;
  cudaStream_t st;
  const char *name;
  ProfScope(const char *n, cudaStream_t s) : st(s), name(n) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (!g_prof.on || g_prof.used + 2 > (int)g_prof.pool.size()) return;
    if (!g_prof.only.empty() && g_prof.only != n) return;
    idx = g_prof.used;
    g_prof.used += 2;
    cudaEventRecord(g_prof.pool[idx], st);
  }
  ~ProfScope() {
    if (idx < 0) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    cudaEventRecord(g_prof.pool[idx + 1], st);
    g_prof.recs.push_back({name, idx, idx + 1});
  }
};

void prof_drain_locked() {
  for (auto &r : g_prof.recs) {
    float ms = 0.f;
    cudaEventSynchronize(g_prof.pool[r.ev1]);
    cudaEventElapsedTime(&ms, g_prof.pool[r.ev0], g_prof.pool[r.ev1]);
    size_t i = 0;
    for (; i < g_prof.names.size(); ++i)
      if (g_prof.names[i] == r.name) break;
    if (i == g_prof.names.size()) {
      g_prof.names.push_back(r.name);
      g_prof.total_ms.push_back(0.0);
      g_prof.count.push_back(0);
    }
    g_prof.total_ms[i] += ms;
    g_prof.count[i] += 1;
  }
  g_prof.recs.clear();
  g_prof.used = 0;
}

#define PROF(name) ProfScope _prof_scope(name, st)

#define CK(expr)                                                                                  \
  do {                                                                                            \
    int _e = (expr);                                                                              \
    if (_e != 0) return fail(GDN_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString((cudaError_t)_e)); \
  } while (0)

// The chunk forward kernel for this problem: tcgen05 for bf16 with d = 128 (its recurrent half, on the
// context that the chunk-local half stored), the mma.sync/CUDA-core kernel otherwise (d = 64, fp32
// inputs, empty batches).
bool tc_forward(const Layout &L, const gdn_shape *s) { return s->dtype == GDN_BF16 && L.D == 128 && L.Ttot > 0; }

// The grid of a tcgen05 recurrent pass (pass 1 / 2 of the forward, the reverse chain).  With equal-length
// sequences whose later segments fit the SMs one CTA each while all segments do not, the later segments take
// one CTA each and the shorter first segments share the remaining SMs, several to a CTA (bal_* in the
// kernel arguments); otherwise one CTA per (segment, head).
dim3 recurrent_grid(const Layout &L, const gdn_shape *s, int &bal_pairs, int &bal_ns, int &bal_big) {
  bal_pairs = bal_ns = bal_big = 0;
  const long slots = num_sms();
  if (!s->cu_seqlens && L.N > 0 && L.S_max % L.N == 0) {
    const long nh = (long)L.N * L.H, ns = L.S_max / L.N;
    if (balanced_plan(nh, (int)ns, slots)) {
      bal_pairs = (int)nh;
      bal_ns = (int)ns;
      bal_big = (int)(nh * (ns - 1));
      return dim3((unsigned)slots);
    }
  }
  return dim3(L.S_max, L.H, 1);
}

// Does the chunk-local half of the tcgen05 forward run in this call and take the gate scan's place (it writes
// the per-chunk gate sums and its last CTA runs the fix-up mode scan)?  Not with the single-launch schedules,
// which the gate scan builds.
bool prep_scans(const Layout &L, const gdn_shape *s) { return tc_forward(L, s) && !single_launch_sp(L, s); }

// plan + gate scan (gate sums to `gsum`), shared by both directions; `scan` false leaves the gate sums and
// the fix-up modes to the chunk-local half (prep_scans)
int prologue(const gdn_shape *s, const Layout &L, char *ws, const float *g, float *gsum, bool scan, cudaStream_t st,
             Plan &pl) {
  pl = plan_of(L, ws);
  int *status = reinterpret_cast<int *>(ws + L.off_status);  // [0] status word, [1]/[2] fix-up flags
  const bool single = single_launch_sp(L, s);
  {
    PROF("plan");
    CK(launch_plan(pl, s->cu_seqlens, L.N, s->cu_seqlens ? s->T : L.Tseq, L.Lseg, L.Lfirst, L.S_max, L.CH_max, status,
                   single ? reinterpret_cast<int *>(ws + L.off_sched) : nullptr, L.sched_zero, st));
  }
  if (scan) {
    PROF("gate_scan");
    const Sched sc[2] = {sched_of(L, ws, 0), sched_of(L, ws, 1)};
    CK(launch_gate_scan(pl, g, L.H, L.CH_max, gsum, status, L.sp ? 1 : 0, L.Lseg, L.Lfirst, L.S_max, s->flags,
                        single ? sc : nullptr, L.N * L.H, st));
  }
  return GDN_OK;
}

// The saved-context backward's prologue: the plan kernel alone, which also runs the fix-up mode scan (and
// builds the schedules) from the gate sums that the forward left in the saved context.
int prologue_saved(const gdn_shape *s, const Layout &L, char *ws, const float *gsum, cudaStream_t st, Plan &pl) {
  pl = plan_of(L, ws);
  int *status = reinterpret_cast<int *>(ws + L.off_status);
  const bool single = single_launch_sp(L, s);
  const Sched sc[2] = {sched_of(L, ws, 0), sched_of(L, ws, 1)};
  PROF("plan");
  CK(launch_plan(pl, s->cu_seqlens, L.N, s->cu_seqlens ? s->T : L.Tseq, L.Lseg, L.Lfirst, L.S_max, L.CH_max, status,
                 single ? reinterpret_cast<int *>(ws + L.off_sched) : nullptr, L.sched_zero, st, gsum, L.H,
                 L.sp ? 1 : 0, s->flags, single ? sc : nullptr));
  return GDN_OK;
}

// ------------------------------------------------------------------ TMA tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [tokens, H, 128] bf16 tensor, box = 64 features x 1 head x 64 tokens, 128-byte swizzle
int qkv_map(CUtensorMap *m, const void *ptr, long tokens, int H) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return GDN_OK;
}

// fp16 per-chunk states [rows, 128] (row-major), box = 64 columns x 128 rows, 128-byte swizzle
int state_map(CUtensorMap *m, const void *ptr, long rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {128, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)rows * 128 * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return GDN_OK;
}

// fp16 tiles [rows, cols], box = 64 columns x `box_rows` rows, 128-byte swizzle (the t64 tiles with
// 64-row boxes, the t128 tiles with 128-row boxes, the 128-column tqkv tiles with 64-row boxes)
int tile_map(CUtensorMap *m, const void *ptr, long rows, int box_rows, int cols = 64) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return GDN_OK;
}
int t64_map(CUtensorMap *m, const Layout &L, const void *ptr) {
  return tile_map(m, ptr, (long)L.CH_max * L.H * T64_TILES * CH, 64);
}
int t128_map(CUtensorMap *m, const Layout &L, const void *ptr) {
  return tile_map(m, ptr, (long)L.CH_max * L.H * T128_TILES * 128, 128);
}
int tqkv_map(CUtensorMap *m, const Layout &L, const void *ptr) {
  return tile_map(m, ptr, (long)L.CH_max * L.H * TQ_TILES * CH, 64, 128);
}
// the reverse chain's tiles, [chunks, H, TC_TILES, 128, 64]: dUt^T (rows d_v, columns token) and the fp16 dO
// (rows 0-63: tokens x features 0-63, rows 64-127: features 64-127), one 128-row box each
int dut_map(CUtensorMap *m, const Layout &L, const void *ptr) {
  return tile_map(m, ptr, (long)L.CH_max * L.H * TC_TILES * 128, 128);
}

int launch_forward_kernel(const Layout &L, const gdn_shape *s, const FwdArgs &fa, dim3 grid, cudaStream_t st) {
  if (tc_forward(L, s)) {
    CUtensorMap t3, tw, ts, tt, to;
    int rc;
    if ((rc = tqkv_map(&t3, L, fa.tqkv)) || (rc = t64_map(&tw, L, fa.t64))) return rc;
    if ((rc = qkv_map(&to, fa.o ? fa.o : fa.k, L.Ttot, L.H))) return rc;  // unused without an output
    // the chunk-start states and W^T, Ut^T tiles written for the backward (maps unused when not saving)
    if ((rc = t128_map(&tt, L, fa.t128 ? fa.t128 : fa.t64))) return rc;
    if ((rc = state_map(&ts, fa.states ? fa.states : fa.k, fa.states ? (long)L.CH_max * L.H * 128 : 128)))
      return rc;
    return launch_fwd_tc(fa, t3, tw, ts, tt, to, grid, st);
  }
  return launch_fwd_chunk(fa, s->dtype == GDN_BF16, L.D, grid, st);
}

// The chunk-local half of the tcgen05 forward: operand tiles, N, P, X1, X2 (and, when the context is
// kept, Ahat and the norms) of every (chunk, head).
int launch_forward_prep(const Layout &L, const FwdArgs &fa, cudaStream_t st) {
  CUtensorMap tq, tk, tv, tw, t3;
  int rc;
  if ((rc = qkv_map(&tk, fa.k, L.Ttot, L.H)) || (rc = qkv_map(&tv, fa.v, L.Ttot, L.H)) ||
      (rc = qkv_map(&tq, fa.q, L.Ttot, L.H)) || (rc = t64_map(&tw, L, fa.t64)) || (rc = tqkv_map(&t3, L, fa.tqkv)))
    return rc;
  return launch_fwd_prep_tc(fa, tq, tk, tv, tw, t3, L.CH_max, st);
}

// Forward state pass: pass A + fix-up when segments exist, then `pass` (1: outputs, 2: states).
int forward_passes(const gdn_shape *s, const Layout &L, char *ws, FwdArgs fa, int pass, cudaStream_t st) {
  if (tc_forward(L, s)) {
    PROF("fwd_prep");
    CK(launch_forward_prep(L, fa, st));
  }
  if (single_launch_sp(L, s)) {  // pass A, the fix-up and pass B in one launch
    fa.pass = pass;
    fa.sched = sched_of(L, ws, 0);
    fa.sched_on = 1;
    PROF(pass == 1 ? "fwd_chunk" : "fwd_states");
    CK(launch_forward_kernel(L, s, fa, dim3(sched_grid(L)), st));
    return GDN_OK;
  }
  if (L.sp) {
    fa.pass = 0;
    {
      PROF("fwd_segment_pass_a");
      dim3 grid(L.S_max, L.H, 2);
      if (tc_forward(L, s)) {  // the (segment, head, role) items by ticket, at most one CTA per SM
        fa.passA_items = 2 * L.S_max * L.H;
        grid = dim3(std::min(fa.passA_items, num_sms()));
      }
      CK(launch_forward_kernel(L, s, fa, grid, st));
      fa.passA_items = 0;
    }
    FixupArgs fx;
    fx.plan = fa.plan;
    fx.gsum = fa.gsum;
    fx.E = fa.Ebuf;
    fx.M = fa.Mbuf;
    fx.out = fa.Sstart;
    fx.H = L.H;
    fx.D = L.D;
    fx.Lseg = L.Lseg;
    fx.Lfirst = L.Lfirst;
    fx.flags = fa.flags;
    fx.reverse = 0;
    fx.fixflag = fa.status + 1;
    fx.status = fa.status;
    fx.ticket = fa.status + 6;  // the row blocks by ticket, at most one CTA per SM
    PROF("fixup_fwd");
    CK(launch_fixup(fx, L.N, num_sms(), st));
  }
  fa.pass = pass;
  dim3 grid(L.S_max, L.H, 1);
  if (tc_forward(L, s)) grid = recurrent_grid(L, s, fa.bal_pairs, fa.bal_ns, fa.bal_big);
  PROF(pass == 1 ? "fwd_chunk" : "fwd_states");
  CK(launch_forward_kernel(L, s, fa, grid, st));
  return GDN_OK;
}

// prep: the chunk-local half writes the gate sums to gsum and scans the fix-up modes (prep_scans)
FwdArgs fwd_args(const gdn_shape *s, const Layout &L, char *ws, const Plan &pl, float *gsum, bool prep) {
  FwdArgs fa;
  std::memset(&fa, 0, sizeof fa);
  fa.plan = pl;
  fa.gsum = gsum;
  if (prep) {
    fa.gsum_out = gsum;
    fa.modes = L.sp ? 1 : 0;
    fa.S_max = L.S_max;
  }
  fa.status = reinterpret_cast<int *>(ws + L.off_status);
  if (L.sp) {
    fa.Ebuf = reinterpret_cast<float *>(ws + L.off_E);
    fa.Mbuf = reinterpret_cast<float *>(ws + L.off_M);
    fa.Sstart = reinterpret_cast<float *>(ws + L.off_S);
  }
  fa.H = L.H;
  fa.Lseg = L.Lseg;
  fa.Lfirst = L.Lfirst;
  fa.scale = s->scale;
  fa.flags = s->flags;
  return fa;
}

int fwd_impl(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g, const float *beta,
             const float *S0, void *o, float *S_T, void *workspace, size_t workspace_bytes, void *saved,
             size_t saved_bytes, gdn_stream_t stream) {
  g_last_error.clear();
  Layout L;
  int rc = make_layout(s, L);
  if (rc) return rc;
  if (L.Ttot > 0 || S_T) {
    rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {g, "g"}, {beta, "beta"}, {o, "o"}},
                    {{S0, "S0"}, {S_T, "S_T"}, {s->cu_seqlens, "cu_seqlens"}});
    if (rc) return rc;
  }
  if (!workspace || workspace_bytes < L.fwd_total)
    return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L.fwd_total,
                workspace ? workspace_bytes : (size_t)0);
  if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  if (saved) {
    if (saved_bytes < L.saved_total)
      return fail(GDN_ERR_WORKSPACE, "saved context of %zu bytes needed, %zu given", L.saved_total, saved_bytes);
    if (!aligned16(saved)) return fail(GDN_ERR_INVALID_ARG, "saved is not 16-byte aligned");
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  // the gate sums go with the saved context, for the saved-context backward
  float *gsum = saved ? reinterpret_cast<float *>(static_cast<char *>(saved) + L.saved_off_gsum)
                      : reinterpret_cast<float *>(ws + L.off_gsum);
  const bool prep = prep_scans(L, s);
  Plan pl;
  if ((rc = prologue(s, L, ws, g, gsum, !prep, st, pl))) return rc;
  FwdArgs fa = fwd_args(s, L, ws, pl, gsum, prep);
  fa.q = q;
  fa.k = k;
  fa.v = v;
  fa.g = g;
  fa.beta = beta;
  fa.S0 = S0;
  fa.o = o;
  fa.ST = S_T;
  if (saved && L.Ttot > 0) {  // the outputs pass also leaves the chunk-start states and context tiles
    fa.states = saved;
    if (L.t64_bytes > 0) {
      fa.t64 = static_cast<char *>(saved) + L.saved_off_t64;
      fa.t128 = static_cast<char *>(saved) + L.saved_off_t128;
      fa.tqkv = static_cast<char *>(saved) + L.saved_off_tqkv;
      fa.nrm = reinterpret_cast<float *>(static_cast<char *>(saved) + L.saved_off_nrm);
    }
  } else if (L.t64_bytes > 0) {  // the two halves of the tcgen05 forward meet in the workspace
    fa.t64 = ws + L.off_fctx_t64;
    fa.tqkv = ws + L.off_fctx_tqkv;
  }
  return forward_passes(s, L, ws, fa, 1, st);
}

int bwd_impl(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g, const float *beta,
             const float *S0, const void *dO, const float *dS_T, void *dq, void *dk, void *dv, float *dg,
             float *dbeta, float *dS0, const void *saved, size_t saved_bytes, void *workspace,
             size_t workspace_bytes, gdn_stream_t stream) {
  g_last_error.clear();
  Layout L;
  int rc = make_layout(s, L);
  if (rc) return rc;
  if (S0 && !dS0) return fail(GDN_ERR_INVALID_ARG, "dS0 is required when S0 is given");
  rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {g, "g"}, {beta, "beta"}, {dO, "dO"}, {dq, "dq"}, {dk, "dk"},
                   {dv, "dv"}, {dg, "dg"}, {dbeta, "dbeta"}},
                  {{S0, "S0"}, {dS_T, "dS_T"}, {dS0, "dS0"}, {s->cu_seqlens, "cu_seqlens"}});
  if (rc) return rc;
  const size_t need = saved ? L.bwd_saved_total : L.bwd_total;
  if (!workspace || workspace_bytes < need)
    return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : (size_t)0);
  if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  if (saved) {
    if (saved_bytes < L.saved_total)
      return fail(GDN_ERR_WORKSPACE, "saved context of %zu bytes needed, %zu given", L.saved_total, saved_bytes);
    if (!aligned16(saved)) return fail(GDN_ERR_INVALID_ARG, "saved is not 16-byte aligned");
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  const bool bf = s->dtype == GDN_BF16;
  Plan pl;
  // the saved-context backward takes the forward's gate sums; the recomputing one forms them again (with its
  // forward's chunk-local half where that runs)
  float *gsum = saved ? reinterpret_cast<float *>(const_cast<char *>(static_cast<const char *>(saved)) +
                                                  L.saved_off_gsum)
                      : reinterpret_cast<float *>(ws + L.off_gsum);
  const bool prep = !saved && prep_scans(L, s);
  if (saved) rc = prologue_saved(s, L, ws, gsum, st, pl);
  else rc = prologue(s, L, ws, g, gsum, !prep, st, pl);
  if (rc) return rc;
  const char *states = ws + L.off_states, *t64 = ws + L.off_t64, *t128 = ws + L.off_t128;
  const char *tqkv = ws + L.off_tqkv, *nrm = ws + L.off_nrm;
  if (saved) {  // the forward left the chunk-start states and context tiles: nothing to recompute
    states = static_cast<const char *>(saved);
    t64 = states + L.saved_off_t64;
    t128 = states + L.saved_off_t128;
    tqkv = states + L.saved_off_tqkv;
    nrm = states + L.saved_off_nrm;
  } else {
    // 1. forward states at every chunk start (and, bf16 with d = 128, the context tiles: a forward
    //    pass that writes no output)
    FwdArgs fa = fwd_args(s, L, ws, pl, gsum, prep);
    fa.q = q;
    fa.k = k;
    fa.v = v;
    fa.g = g;
    fa.beta = beta;
    fa.S0 = S0;
    fa.states = ws + L.off_states;
    const bool tiles = L.t64_bytes > 0 && L.Ttot > 0;
    if (tiles) {
      fa.t64 = ws + L.off_t64;
      fa.t128 = ws + L.off_t128;
      fa.tqkv = ws + L.off_tqkv;
      fa.nrm = reinterpret_cast<float *>(ws + L.off_nrm);
    }
    if ((rc = forward_passes(s, L, ws, fa, tiles ? 1 : 2, st))) return rc;
  }
  // 2. reverse chain: dS at every chunk end (and dS0)
  BwdArgs ba;
  std::memset(&ba, 0, sizeof ba);
  ba.q = q;
  ba.k = k;
  ba.v = v;
  ba.dO = dO;
  ba.g = g;
  ba.beta = beta;
  ba.dST = dS_T;
  ba.dq = dq;
  ba.dk = dk;
  ba.dv = dv;
  ba.dg = dg;
  ba.dbeta = dbeta;
  ba.dS0 = dS0;
  ba.plan = pl;
  ba.gsum = gsum;
  ba.status = reinterpret_cast<int *>(ws + L.off_status);
  if (L.sp) {
    ba.Fbuf = reinterpret_cast<float *>(ws + L.off_F);
    ba.Rbuf = reinterpret_cast<float *>(ws + L.off_R);
    ba.dSend = reinterpret_cast<float *>(ws + L.off_dS);
  }
  ba.states = states;
  ba.nrm = reinterpret_cast<const float *>(nrm);
  ba.dstates = ws + L.off_dstates;
  ba.H = L.H;
  ba.Lseg = L.Lseg;
  ba.Lfirst = L.Lfirst;
  if (!s->cu_seqlens && L.Tseq > 0) {  // equal-length sequences: the local kernel's chunk order
    ba.ord_n = L.N;
    ba.ord_nc = (L.Tseq + CH - 1) / CH;
  }
  ba.scale = s->scale;
  ba.flags = s->flags;
  // the reverse chain: tcgen05 for bf16 with d = 128, the mma.sync kernel otherwise
  const bool chain_tc = bf && L.D == 128 && L.Ttot > 0;
  CUtensorMap cmaps[6];
  if (chain_tc && ((rc = tqkv_map(&cmaps[0], L, tqkv)) || (rc = qkv_map(&cmaps[1], dO, L.Ttot, L.H)) ||
                   (rc = t64_map(&cmaps[2], L, t64)) || (rc = t128_map(&cmaps[3], L, t128)) ||
                   (rc = state_map(&cmaps[4], ba.dstates, (long)L.CH_max * L.H * 128)) ||
                   (rc = dut_map(&cmaps[5], L, ws + L.off_dut))))
    return rc;
  auto chain = [&](dim3 grid) {
    return chain_tc ? launch_bwd_chain_tc(ba, cmaps, grid, st) : launch_bwd_chain(ba, bf, L.D, grid, st);
  };
  if (single_launch_sp(L, s) && chain_tc) {  // pass A, the fix-up and the chain in one launch
    ba.pass = 1;
    ba.sched = sched_of(L, ws, 1);
    ba.sched_on = 1;
    PROF("bwd_chain");
    CK(chain(dim3(sched_grid(L))));
  } else {
  if (L.sp) {
    ba.pass = 0;
    {
      PROF("bwd_chain_pass_a");
      dim3 grid(L.S_max, L.H, 2);
      if (chain_tc) {  // the (segment, head, role) items by ticket, at most one CTA per SM
        ba.passA_items = 2 * L.S_max * L.H;
        grid = dim3(std::min(ba.passA_items, num_sms()));
      }
      CK(chain(grid));
      ba.passA_items = 0;
    }
    FixupArgs fx;
    fx.plan = pl;
    fx.gsum = ba.gsum;
    fx.E = ba.Fbuf;
    fx.M = ba.Rbuf;
    fx.out = ba.dSend;
    fx.H = L.H;
    fx.D = L.D;
    fx.Lseg = L.Lseg;
    fx.Lfirst = L.Lfirst;
    fx.flags = s->flags;
    fx.reverse = 1;
    fx.fixflag = ba.status + 2;
    fx.status = ba.status;
    fx.ticket = ba.status + 7;  // the row blocks by ticket, at most one CTA per SM
    PROF("fixup_bwd");
    CK(launch_fixup(fx, L.N, num_sms(), st));
  }
  ba.pass = 1;
  {
    dim3 grid(L.S_max, L.H, 1);
    if (chain_tc) grid = recurrent_grid(L, s, ba.bal_pairs, ba.bal_ns, ba.bal_big);
    PROF("bwd_chain");
    CK(chain(grid));
  }
  }
  // 3. local gradients, every (chunk, head) in parallel
  {
    PROF("bwd_local");
    if (bf && L.D == 128 && L.Ttot > 0) {
      CUtensorMap maps[9];
      if ((rc = tqkv_map(&maps[0], L, tqkv)) || (rc = dut_map(&maps[1], L, ws + L.off_dut)) ||
          (rc = state_map(&maps[2], states, (long)L.CH_max * L.H * 128)) ||
          (rc = state_map(&maps[3], ws + L.off_dstates, (long)L.CH_max * L.H * 128)) ||
          (rc = t64_map(&maps[4], L, t64)) || (rc = qkv_map(&maps[5], dq, L.Ttot, L.H)) ||
          (rc = qkv_map(&maps[6], dk, L.Ttot, L.H)) || (rc = qkv_map(&maps[7], dv, L.Ttot, L.H)) ||
          (rc = t128_map(&maps[8], L, t128)))
        return rc;
      CK(launch_bwd_local_tc(ba, maps, L.CH_max, st));
    } else {
      CK(launch_bwd_local(ba, bf, L.D, L.CH_max, st));
    }
  }
  return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_fwd_workspace_size(const gdn_shape *shape) {
  Layout L;
  if (make_layout(shape, L) != GDN_OK) return 0;
  return L.fwd_total;
}

size_t gdn_bwd_workspace_size(const gdn_shape *shape) {
  Layout L;
  if (make_layout(shape, L) != GDN_OK) return 0;
  return L.bwd_total;
}

size_t gdn_saved_size(const gdn_shape *shape) {
  Layout L;
  if (make_layout(shape, L) != GDN_OK) return 0;
  return L.saved_total;
}

size_t gdn_bwd_saved_workspace_size(const gdn_shape *shape) {
  Layout L;
  if (make_layout(shape, L) != GDN_OK) return 0;
  return L.bwd_saved_total;
}

int gdn_chunk_fwd(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const float *S0, void *o, float *S_T, void *workspace, size_t workspace_bytes,
                  gdn_stream_t stream) {
  return fwd_impl(s, q, k, v, g, beta, S0, o, S_T, workspace, workspace_bytes, nullptr, 0, stream);
}

int gdn_chunk_fwd_save(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const float *S0, void *o, float *S_T, void *saved, size_t saved_bytes,
                       void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
  if (!saved) {
    g_last_error.clear();
    return fail(GDN_ERR_INVALID_ARG, "saved is NULL (use gdn_chunk_fwd to save nothing)");
  }
  return fwd_impl(s, q, k, v, g, beta, S0, o, S_T, workspace, workspace_bytes, saved, saved_bytes, stream);
}

}  // extern "C"

// ------------------------------------------------------------ no-allocation forward
// Scratch for gdn_chunk_fwd_static: a fixed array in device memory that every
// GPU loading this library holds until the process exits.  Host code only sees
// a host-side stand-in under this name; its device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
namespace {
constexpr size_t kStaticScratchBytes = (size_t)GDN_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
}  // namespace

extern "C" {

int gdn_chunk_fwd_static(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                         const float *beta, const float *S0, void *o, float *S_T, gdn_stream_t stream) {
  g_last_error.clear();
  Layout L;
  int rc = make_layout(s, L);
  if (rc) return rc;
  gdn_shape sh = *s;
  if (L.fwd_total > kStaticScratchBytes && !(sh.flags & GDN_SP_OFF)) {
    // the sequence-parallel buffers do not fit: run one segment per sequence
    sh.flags |= GDN_SP_OFF;
    if ((rc = make_layout(&sh, L))) return rc;
  }
  if (L.fwd_total > kStaticScratchBytes)
    return fail(GDN_ERR_WORKSPACE,
                "gdn_chunk_fwd_static: this shape needs %zu bytes of scratch, the static scratch holds %zu "
                "(use gdn_chunk_fwd with a caller-provided workspace)",
                L.fwd_total, kStaticScratchBytes);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(GDN_ERR_CUDA, "gdn_chunk_fwd_static: no usable current device");
  void *ptr = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
      // the address lookup may not run inside a stream capture: refuse that case with a clear message
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) != cudaSuccess)
        return fail(GDN_ERR_CUDA, "gdn_chunk_fwd_static: cudaStreamIsCapturing failed");
      if (cs != cudaStreamCaptureStatusNone)
        return fail(GDN_ERR_INVALID_ARG,
                    "gdn_chunk_fwd_static: the first call on device %d must come before any stream capture "
                    "(it looks up the static scratch's device address)", dev);
      void *p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess || !p)
        return fail(GDN_ERR_CUDA, "gdn_chunk_fwd_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      g_static_ptr[dev] = p;
    }
    ptr = g_static_ptr[dev];
  }
  return gdn_chunk_fwd(&sh, q, k, v, g, beta, S0, o, S_T, ptr, kStaticScratchBytes, stream);
}

int gdn_chunk_bwd(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const float *S0, const void *dO, const float *dS_T, void *dq, void *dk, void *dv, float *dg,
                  float *dbeta, float *dS0, void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
  return bwd_impl(s, q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, nullptr, 0, workspace,
                  workspace_bytes, stream);
}

int gdn_chunk_bwd_saved(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *S0, const void *dO, const float *dS_T, void *dq, void *dk,
                        void *dv, float *dg, float *dbeta, float *dS0, const void *saved, size_t saved_bytes,
                        void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
  if (!saved) {
    g_last_error.clear();
    return fail(GDN_ERR_INVALID_ARG, "saved is NULL (use gdn_chunk_bwd to recompute the forward)");
  }
  return bwd_impl(s, q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, saved, saved_bytes, workspace,
                  workspace_bytes, stream);
}
int gdn_recurrent_fwd(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                      const float *beta, const float *S_in, void *o, float *S_out, gdn_stream_t stream) {
  g_last_error.clear();
  if (!s) return fail(GDN_ERR_INVALID_ARG, "shape is NULL");
  if (s->reserved[0] || s->reserved[1]) return fail(GDN_ERR_INVALID_ARG, "reserved fields must be 0");
  if (s->B < 1 || s->T < 0 || s->H < 1) return fail(GDN_ERR_INVALID_ARG, "need B >= 1, T >= 0, H >= 1");
  if (s->cu_seqlens) return fail(GDN_ERR_UNSUPPORTED, "the recurrent form takes B sequences of T tokens (cu_seqlens must be NULL)");
  if (s->Dk != s->Dv) return fail(GDN_ERR_UNSUPPORTED, "d_k != d_v is not supported");
  if (s->Dk != 64 && s->Dk != 128) return fail(GDN_ERR_UNSUPPORTED, "d must be 64 or 128 (got %d)", s->Dk);
  if (s->dtype != GDN_BF16 && s->dtype != GDN_FP32) return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
  if (!std::isfinite(s->scale) || s->scale == 0.f) return fail(GDN_ERR_INVALID_ARG, "scale must be finite and non-zero");
  if ((long)s->B * s->H > (long)INT32_MAX / 4 || (long)s->B * s->T > (long)INT32_MAX / 2)
    return fail(GDN_ERR_UNSUPPORTED, "too many sequences or tokens");
  int rc = check_ptrs({{S_out, "S_out"}}, {{S_in, "S_in"}});
  if (rc) return rc;
  if (s->T > 0 && (rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {g, "g"}, {beta, "beta"}, {o, "o"}}, {})))
    return rc;
  RecArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.S_in = S_in;
  a.o = o;
  a.S_out = S_out;
  a.T = s->T;
  a.H = s->H;
  a.scale = s->scale;
  a.flags = s->flags;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  PROF("recurrent");
  CK(launch_recurrent(a, s->dtype == GDN_BF16, s->Dk, s->B * s->H, st));
  return GDN_OK;
}

int gdn_get_device_status(const gdn_shape *shape, const void *workspace, gdn_stream_t stream) {
  (void)shape;
  int v = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // workspace NULL: the status word of gdn_chunk_fwd_static, word 0 of the static scratch on the
  // current device (read through the symbol, so no cached address is involved)
  const cudaError_t e = workspace ? cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st)
                                  : cudaMemcpyFromSymbolAsync(&v, g_static_scratch, 4, 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  return v;
}

int gdn_device_status_code(int word) {
  if (word < 0) return GDN_ERR_CUDA;
  if (word & 2) return GDN_ERR_INVALID_ARG;
  if (word & (4 | 8 | 16)) return GDN_ERR_TIMEOUT;
  if (word & 1) return GDN_ERR_NUMERIC;
  return GDN_OK;
}

int gdn_plan_estimate(const gdn_shape *shape, double *fwd_us, double *bwd_us) {
  Layout L;
  int rc = make_layout(shape, L);
  if (rc) return rc;
  const int maxc = shape->cu_seqlens ? (int)((L.Ttot + CH - 1) / CH) : (shape->T + CH - 1) / CH;
  double f = 0.0, b = 0.0;
  if (maxc > 0) plan_cost_us(*shape, L.N, maxc, L.CH_max, std::min(L.Lseg, maxc), std::min(L.Lfirst, maxc), &f, &b);
  if (fwd_us) *fwd_us = f;
  if (bwd_us) *bwd_us = b;
  return GDN_OK;
}

int gdn_plan_query(const gdn_shape *shape, int *seg_chunks, int *max_segments, int *max_chunks, int *seg_first) {
  Layout L;
  int rc = make_layout(shape, L);
  if (rc) return rc;
  if (seg_chunks) *seg_chunks = L.Lseg;
  if (seg_first) *seg_first = L.Lfirst;
  if (max_segments) *max_segments = L.S_max;
  if (max_chunks) *max_chunks = L.CH_max;
  return GDN_OK;
}

int gdn_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (on && g_prof.pool.empty()) {
    g_prof.pool.resize(8192);
    for (auto &e : g_prof.pool)
      if (cudaEventCreate(&e) != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaEventCreate failed");
  }
  if (!on) prof_drain_locked();
  g_prof.on = on != 0;
  return GDN_OK;
}

int gdn_profile_only(const char *name) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.only = name ? name : "";
  return GDN_OK;
}

int gdn_profile_report(char *buf, size_t len, int reset) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  prof_drain_locked();
  std::string out;
  char line[256];
  for (size_t i = 0; i < g_prof.names.size(); ++i) {
    snprintf(line, sizeof line, "%s %ld %.6f\n", g_prof.names[i].c_str(), g_prof.count[i], g_prof.total_ms[i]);
    out += line;
  }
  if (reset) {
    g_prof.names.clear();
    g_prof.total_ms.clear();
    g_prof.count.clear();
  }
  if (buf && len) {
    const size_t n = std::min(len - 1, out.size());
    memcpy(buf, out.data(), n);
    buf[n] = 0;
  }
  return (int)out.size();
}

const char *gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    case GDN_ERR_CUDA: return "CUDA error";
    case GDN_ERR_TIMEOUT: return "a bounded device wait expired";
    case GDN_ERR_NUMERIC: return "an fp16 tensor-core operand overflowed or was not finite";
    default: return "unknown status";
  }
}

const char *gdn_last_error_string(void) { return g_last_error.c_str(); }

}  // extern "C"
