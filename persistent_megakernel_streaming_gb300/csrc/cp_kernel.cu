// cp_kernel.cu -- the frame kernel for sm_103a.
//
// One CTA per SM walks its static task list ("Qwen3-TTS: Run the 1.7B Depth
// Loop as One Persistent Kernel on Hopper", section "How it works"). The CTA
// is warp-specialised:
//   warp 0     streams every projection task's weights, in list order, into a
//              ring of shared-memory pages with bulk (TMA) copies. Weights never
//              depend on activations, so it runs ahead of every dependency wait
//              as far as the ring allows ("The gaps between kernels: PDL and
//              megakernels", section "Megakernels": prefetching across kernels).
//   warp 1     issues tcgen05 MMAs: D[64 rows x N features] in TMEM +=
//              A[activation K-chunk] * B[weight K-chunk]^T, bf16 in, fp32 acc.
//   warps 2-9  wait on dependency counters, stage activations into the A slots
//              (bf16 chunks as their producers wrote them), read the accumulator,
//              exchange K-split partial sums with the cluster through
//              distributed shared memory, run the epilogues, attention and the
//              draw, store, and signal counters.
// A projection tile is split along K over the C CTAs of a cluster; each CTA
// sends its partial rows to the CTA that owns them, which adds the C partials
// in rank order (fixed order, no atomics: the frame is bit-identical run to
// run, as in section "How it works" for the o/down split).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <curand_philox4x32_x.h>

#include "cp.h"
#include "cp_internal.h"
#include "cp_ptx.cuh"

// The file is built three times: as is (every size read from the kernel
// parameters) and with CP_SHAPE_1P7B defined, which fixes the sizes in
// kShape1p7b at compile time, once for handles of up to 64 rows (M = 64
// projections) and once, with CP_ROWS_128, for handles of more (M = 128).
// The compiler then folds them into the addressing and drops the branches
// that shape never takes (a 64-row frame measured 7.8 % faster); the host
// picks the build per handle. The test kernels live in the generic build only.
#ifdef CP_SHAPE_1P7B
#ifdef CP_ROWS_128
#define CP_BUILD cp17r128
#else
#define CP_BUILD cp17
#endif
#else
#define CP_BUILD generic
#endif

namespace cp {
namespace CP_BUILD {
using namespace ptx;

// The shape and cluster size this build runs with.
__device__ __forceinline__ Shape shape_of(const KParams& p) {
  Shape s = p.s;
#ifdef CP_SHAPE_1P7B
  s.L = kShape1p7b.L; s.H = kShape1p7b.H; s.Hq = kShape1p7b.Hq; s.Hkv = kShape1p7b.Hkv; s.D = kShape1p7b.D;
  s.F = kShape1p7b.F; s.P = kShape1p7b.P; s.V = kShape1p7b.V; s.T = kShape1p7b.T; s.qk_norm = kShape1p7b.qk_norm;
#endif
  return s;
}
__device__ __forceinline__ int cluster_of(const KParams& p) {
#ifdef CP_SHAPE_1P7B
  return kShape1p7b.cluster;
#else
  return p.cluster;
#endif
}
// Rows per projection MMA: 64, or 128 for a handle of more than 64 rows. An
// M = 128 handle stages each activation K-chunk into two adjacent A slots
// (16 KB, one 128-row operand), so kNumA / 2 chunks are in flight, and its
// partial-sum exchange uses the two receive slots as one.
__device__ __forceinline__ bool m128_of(const KParams& p) {
#ifdef CP_SHAPE_1P7B
#ifdef CP_ROWS_128
  return true;
#else
  return false;
#endif
#else
  return p.m128 != 0;
#endif
}
// A chunk slots of the handle's mode (8 of 64 rows or 4 of 128), log2.
__device__ __forceinline__ int a_log2(const KParams& p) { return m128_of(p) ? 2 : 3; }

constexpr int kNumAcc = 2;       // TMEM accumulators (a two-tile task holds both)
constexpr int kAccCols = 256;    // columns per accumulator (tiles up to N = 256)

// Barrier slots in the misc region.
enum {
  B_WFULL = 0,
  B_WEMPTY = B_WFULL + kNumW,
  B_AFULL = B_WEMPTY + kNumW,
  B_AEMPTY = B_AFULL + kNumA,
  B_ACCFULL = B_AEMPTY + kNumA,
  B_ACCEMPTY = B_ACCFULL + kNumAcc,
  B_RFULL = B_ACCEMPTY + kNumAcc,
  B_RFREE = B_RFULL + 2,
  B_DRAIN = B_RFREE + 2,
  B_SCR = B_DRAIN + 1,   // bulk copies into the scratch area (attention's keys and values)
  B_COUNT = B_SCR + 1
};
static_assert(B_COUNT * 8 <= 512, "barrier area");
constexpr int kMiscTmem = 512;   // u32: TMEM base address
constexpr int kMiscFlag = 516;   // i32 flags
constexpr int kMiscEarly = 524;  // u32: the current attention task's early copy was issued
constexpr int kMiscTask = 640;   // two Task records: the compute warps' current and next task
static_assert(kMiscTask + 2 * (int)sizeof(Task) <= kSmemMiscBytes, "misc area");
constexpr int kTmemCols = kNumAcc * kAccCols;
static_assert(kTmemCols <= 512 && kMaxTileN <= kAccCols, "TMEM accumulators");

struct Sm {
  uint8_t* base;
  uint32_t b;  // shared address of base
  __device__ uint32_t bar(int i) const { return b + kSmemMisc + i * 8; }
  __device__ uint32_t a_slot(int s) const { return b + kSmemA + s * kAChunkBytes; }
  // A chunk slot `s` of a handle whose chunks are `m128` ? 128 : 64 rows
  __device__ uint32_t a_chunk(int s, bool m128) const { return b + kSmemA + (s << (m128 ? 14 : 13)); }
  __device__ uint32_t w_page(int s) const { return b + kSmemW + s * kPageBytes; }
  __device__ uint32_t recv(int s) const { return b + kSmemRecv + s * kRecvBytes; }
  __device__ float* recv_ptr(int s) const { return reinterpret_cast<float*>(base + kSmemRecv + s * kRecvBytes); }
  __device__ uint32_t* misc_u32(int off) const { return reinterpret_cast<uint32_t*>(base + kSmemMisc + off); }
  __device__ uint8_t* scratch() const { return base + kSmemA; }  // A slots double as scratch outside projections
};

// ---------------------------------------------------------------- status
__device__ __forceinline__ bool aborted(const KParams& p) {
  return *reinterpret_cast<volatile int32_t*>(p.status + 1) != 0;
}
__device__ __noinline__ void raise_error(const KParams& p, int code, int detail) {
  if (atomicCAS(p.status, 0, code) == 0) {
    p.status[3] = detail;
    p.status[4] = blockIdx.x;
  }
  atomicExch(p.status + 1, 1);
}

// Bounded waits: give up on abort or after the timeout (setting the status).
// They spin on test_wait (no suspension): the frame is a latency chain and a
// suspended waiter wakes later than the phase completes. The spin loops are
// inlined: out of line, each call saved and restored registers through local
// memory, and with the L1 this small (218 KB of the SM's memory is shared
// memory) the restore at the end of a wait usually went to L2, right on the
// critical path (measured: the frame 3.5 % faster inlined).
// A wait reads the global abort flag only once it has lasted kAbortCheckNs:
// the read is an L2 round trip, and a phase completing during it would be
// seen that much later (waits in a running frame are shorter than that).
// With `backoff` a waiter that has probed for a while (about half a
// microsecond) sleeps between probes: long waits of the compute warps then
// leave issue slots to the MMA and producer warps, short ones are not
// lengthened by a sleep (the MMA warp itself polls without sleeping).
constexpr uint64_t kAbortCheckNs = 20000;
__device__ __forceinline__ bool wait_bar_slow(const KParams& p, uint32_t bar, uint32_t parity, int where, bool cluster,
                                           bool backoff) {
  const uint64_t t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (cluster ? mb_test_cluster(bar, parity) : mb_test(bar, parity)) return true;
    if (backoff && i > 32) __nanosleep(64);
    if ((i & 63) == 0) {
      const uint64_t dt = gtime() - t0;
      if (dt > kAbortCheckNs && aborted(p)) return false;
      if (dt > (uint64_t)p.timeout_ns) {
        raise_error(p, CP_ERR_TIMEOUT, where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bar(const KParams& p, uint32_t bar, uint32_t parity, int where,
                                         bool cluster = false, bool backoff = false) {
  if (cluster ? mb_test_cluster(bar, parity) : mb_test(bar, parity)) return true;
  return wait_bar_slow(p, bar, parity, where, cluster, backoff);
}
// Warp-collective wait: lane 0 polls, the warp then synchronises (ordering its
// lanes' later accesses after the wait) and shares the result, so a waiting
// CTA does not flood the shared-memory pipe with 256 pollers.
__device__ __forceinline__ bool wait_bar_w(const KParams& p, uint32_t bar, uint32_t parity, int where,
                                           bool cluster = false) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(p, bar, parity, where, cluster, true);
  __syncwarp();
  return __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
}
// Drain wait used at teardown: ignores the abort flag, still bounded.
__device__ __noinline__ void drain_bar(const KParams& p, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gtime();
  while (!mb_try(bar, parity)) {
    if (gtime() - t0 > (uint64_t)p.timeout_ns) {
      raise_error(p, CP_ERR_TIMEOUT, 0x7000);
      return;
    }
  }
}
__device__ __forceinline__ bool wait_counter(const KParams& p, int idx, uint32_t target, int where) {
  const uint32_t* c = p.counters + idx;
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire(c) >= target) return true;
    if ((i & 15) == 0) {
      const uint64_t dt = gtime() - t0;
      if (dt > kAbortCheckNs && aborted(p)) return false;
      if (dt > (uint64_t)p.timeout_ns) {
        raise_error(p, CP_ERR_TIMEOUT, where);
        return false;
      }
    }
  }
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
// Two floats rounded to bf16 (nearest even), a in the low half: one cvt.
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).
__device__ __forceinline__ uint4 philox10(uint4 c, uint2 k) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}
// (word >> 9 + 0.5) * 2^-23: exact in fp32, strictly inside (0, 1).
__device__ __forceinline__ float philox_uniform(uint32_t w) {
  return ((float)(w >> 9) + 0.5f) * 1.1920928955078125e-07f;
}

// ---------------------------------------------------------------- per-thread state
struct CState {
  uint32_t a_it, acc_it, recv_it;
  uint32_t w_it;    // weight pages of the projection tasks so far (mirrors the MMA warp's count)
  uint32_t scr_it;  // uses of the scratch barrier (leader issues, every thread waits)
  int gidx;         // global index of the task being run (trace only)
  uint32_t a_bulk;  // bit s: slot s's latest use was a bulk copy (leader only; teardown drain)
};

__device__ __forceinline__ void trace_stamp(const KParams& p, int gidx, int s) {
  if (p.trace) p.trace[(size_t)gidx * kTraceStamps + s] = (int64_t)gtime();
}

// Signal: one barrier over the compute warps (every store of this CTA's task
// is then ordered before the leader's release, as in a grid barrier), then
// one release-add on the counter. Returns false if any compute thread failed.
__device__ __forceinline__ bool finish_and_signal(const KParams& p, const Task& t, int ct, int gidx, bool ok) {
  if (ct == 0) cp_async_wait_all();  // the next task's record (compute_role) has landed
  if (csync_or(!ok)) return false;
  if (ct == 0) {
    trace_stamp(p, gidx, 5);
    if (p.mode == 0) red_release_add(p.counters + t.signal, 1);
    trace_stamp(p, gidx, 6);
  }
  return true;
}

__device__ bool task_wait(const KParams& p, const Task& t, int ct, int gidx) {
  bool ok = true;
  if (ct == 0) {
    trace_stamp(p, gidx, 0);
    if (p.trace)
      p.trace[(size_t)gidx * kTraceStamps + 7] = ((int64_t)t.phase << 32) | ((int64_t)t.kind << 16) | blockIdx.x;
    if (p.mode == 0) {
      if (gidx == p.stall_task) ok = wait_counter(p, 0, 0x40000000u, 0x1FFF);  // testing: a count nothing reaches
      if (ok && t.wait0 >= 0) ok = wait_counter(p, t.wait0, (uint32_t)t.target0, 0x1000 + t.phase);
      // an attention task's second counter only guards its early copy (see attn_task)
      if (ok && t.wait1 >= 0 && t.type != T_ATTN) ok = wait_counter(p, t.wait1, (uint32_t)t.target1, 0x1000 + t.phase);
    }
    trace_stamp(p, gidx, 1);
  }
  return !csync_or(!ok);
}

// ---------------------------------------------------------------- projection
// Stage one K part of the talker hidden state (fp32, the input projection's
// operand) into A slots as bf16 in the 128-byte swizzle layout: row r's
// 16-byte unit u sits at unit u ^ (r & 7). Thread ct handles row ct/4 (and
// 64 + ct/4 in an M = 128 handle) and 16 consecutive K elements of each
// chunk; up to four (chunk, 64-row half) pieces are loaded at once. After the
// stores every thread fences for the async proxy, the compute warps meet, and
// the leader arrives on each chunk's full barrier. Returns false if a wait
// failed (abort).
__device__ bool stage_rows(const KParams& p, const Task& t, const FrameArgs& fa, Sm sm, CState& st, int ct,
                           const float* src, int ld) {
  const int R = fa.rows;
  const bool m128 = m128_of(p);
  const int nh = m128 ? 2 : 1, per = 4 / nh, lg = a_log2(p), nA = 1 << lg;
  const int seg = ct & 3;
  bool ok = true;
  for (int kb = 0; kb < t.nkc; kb += per) {
    const int nb = min(per, t.nkc - kb);
    float4 xv[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = q / nh, row = (q % nh) * 64 + (ct >> 2);
      const int k = t.k0 + (kb + c) * 64 + seg * 16;
      if (c < nb && row < R) {
        const float4* xp = reinterpret_cast<const float4*>(src + (size_t)row * ld + k);
#pragma unroll
        for (int e = 0; e < 4; ++e) xv[q][e] = xp[e];
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) xv[q][e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c < nb && ok) {
        const uint32_t it = st.a_it + kb + c;
        ok = wait_bar_w(p, sm.bar(B_AEMPTY + (it & (nA - 1))), ((it >> lg) & 1) ^ 1, 0x2000);
      }
    if (ok) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = q / nh, row = (q % nh) * 64 + (ct >> 2);
        if (c < nb && row < R) {
          const float x[16] = {xv[q][0].x, xv[q][0].y, xv[q][0].z, xv[q][0].w, xv[q][1].x, xv[q][1].y,
                               xv[q][1].z, xv[q][1].w, xv[q][2].x, xv[q][2].y, xv[q][2].z, xv[q][2].w,
                               xv[q][3].x, xv[q][3].y, xv[q][3].z, xv[q][3].w};
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) pk[i] = pack_bf2(x[2 * i], x[2 * i + 1]);
          const uint32_t rb = sm.a_chunk((int)((st.a_it + kb + c) & (nA - 1)), m128) + row * 128;
          st_shared_v4u(rb + (((seg * 2 + 0) ^ (row & 7)) << 4), make_uint4(pk[0], pk[1], pk[2], pk[3]));
          st_shared_v4u(rb + (((seg * 2 + 1) ^ (row & 7)) << 4), make_uint4(pk[4], pk[5], pk[6], pk[7]));
        }
      }
    }
    fence_proxy_async_smem();
    ok = !csync_or(!ok);
    if (ct == 0 && ok)
      for (int c = 0; c < nb; ++c) mb_arrive(sm.bar(B_AFULL + ((st.a_it + kb + c) & (nA - 1))));
  }
  st.a_it += t.nkc;
  return ok;
}

// Per-chunk wait ("What's left in the frame, open": a projection starts each
// K chunk as soon as the producer tiles of that chunk are done): input chunk
// c of the task's K part (64 elements from k0 + 64 c) waits for the counter
// slots its producers signal, (k0 + 64 c) / fps .. (k0 + 64 c + 63) / fps of
// the producer phase (fps: input features per slot). Bounded like every wait.
__device__ __forceinline__ bool chunk_wait(const KParams& p, const Task& t, int c) {
  const int fps = t.cpack >> 16;
  const uint32_t tg = (uint32_t)(t.cpack & 0xFFFF);
  const int e0 = t.k0 + 64 * c;
  for (int sl = e0 / fps; sl <= (e0 + 63) / fps; ++sl)
    if (!wait_counter(p, t.cbase + sl, tg, 0x1000 + t.phase)) return false;
  return true;
}

// Stage a K part already stored as bf16 128-byte-swizzled chunks [chunk][row]
// (x times its norm gain, the attention output, the SwiGLU output) with one
// bulk copy of the R live rows per chunk, expect-tx on the chunk's full
// barrier; the MMA warp starts on a chunk as soon as it lands. The first
// round (up to one chunk per slot: 8, or 4 in an M = 128 handle) is issued by
// lanes of the leader's warp, one chunk each, and with per-chunk waits each
// lane first polls its own chunk's producers: issued by one thread, a task's
// copies landed one after another (measured ~0.4 us apart; one lane per copy:
// the frame 2.7 % faster). A slot's previous use in an earlier task was
// released by the leader itself (release_inputs, after that task's
// accumulator, so its MMAs had read it): only refills within the task (down:
// 12 chunks through 8 slots) wait, for the MMA warp's commit; their chunks'
// producers are polled by one lane each right after the first round, and the
// leader issues the refills. The leader also keeps the bookkeeping of every
// copy (the teardown drain after an abort). Returns false on abort, uniformly
// for the leader's warp.
__device__ bool stage_chunks(const KParams& p, const Task& t, const FrameArgs& fa, Sm sm, CState& st, int ct,
                             const uint16_t* chunks) {
  bool ok = true;
  if (ct < 32) {
    if (ct == 0 && p.stall_staging && p.mode == 0) ok = wait_counter(p, 0, 0x40000000u, 0x2FFF);  // testing
    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    const bool m128 = m128_of(p);
    const int lg = a_log2(p), nA = 1 << lg;
    const uint32_t a0 = st.a_it;
    const int n1 = min(t.nkc, nA);
    const uint32_t bytes = (uint32_t)fa.rows * 128u;
    const size_t cbytes = (size_t)shape_of(p).MR * 128;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(chunks) + (size_t)(t.k0 / 64) * cbytes;
    // first round: lane c takes chunk c; with per-chunk waits it polls that
    // chunk's producers itself, so each copy leaves as soon as its own input
    // is done (the lanes poll side by side)
    const bool chunked = t.cbase >= 0 && p.mode == 0;
    bool lok = ok;
    if (ok && ct < n1) {
      if (chunked) {
        lok = chunk_wait(p, t, ct);
        if (ct == 0) trace_stamp(p, st.gidx, 1);  // the first chunk's dependency seen
      }
      if (lok) {
        fence_proxy_async_global();
        const int slot = (int)((a0 + (uint32_t)ct) & (nA - 1));
        mb_expect(sm.bar(B_AFULL + slot), bytes);
        bulk_g2s(sm.a_chunk(slot, m128), src + (size_t)ct * cbytes, bytes, sm.bar(B_AFULL + slot));
      }
    }
    const uint32_t issued = __ballot_sync(0xffffffffu, ok && lok && ct < n1);
    ok = __all_sync(0xffffffffu, lok);
    // the chunks beyond the first round (refills through freed slots): their
    // producers are polled now, one lane each, side by side, while the first
    // chunks' MMAs run; the leader's refills then only wait for free slots
    if (chunked && ok && t.nkc > n1) {
      bool rok = true;
      for (int c = n1 + ct; c < t.nkc; c += 32) rok = rok && chunk_wait(p, t, c);
      ok = __all_sync(0xffffffffu, rok);
    }
    if (ct == 0) {
      // the teardown drain waits for each slot's latest bulk copy: mark the
      // ones that left, and unmark the slots of copies that never did
      for (int c = 0; c < n1; ++c) {
        const uint32_t bit = 1u << ((a0 + (uint32_t)c) & (nA - 1));
        st.a_bulk = (issued >> c) & 1u ? (st.a_bulk | bit) : (st.a_bulk & ~bit);
      }
      // (the first round is accounted for, issued or not: the drain reads a_bulk)
      int kc = n1;
      for (; ok && kc < t.nkc; ++kc) {
        const uint32_t it = a0 + (uint32_t)kc;
        const int slot = (int)(it & (nA - 1));
        ok = wait_bar(p, sm.bar(B_AEMPTY + slot), ((it >> lg) & 1) ^ 1, 0x2100);
        if (!ok) break;
        mb_expect(sm.bar(B_AFULL + slot), bytes);
        bulk_g2s(sm.a_chunk(slot, m128), src + (size_t)kc * cbytes, bytes, sm.bar(B_AFULL + slot));
        st.a_bulk |= 1u << slot;
      }
      // after an abort the leader's count covers only what was issued, so the
      // teardown drain names each slot's latest copy and none that never left
      if (!ok) st.a_it = a0 + (uint32_t)kc;
    }
    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    if (!ok) return false;
  }
  st.a_it += t.nkc;
  return ok;
}

// One 16-byte piece of a K-split partial into its owner's receive slot: a
// peer's through the cluster, counted in bytes on the owner's receive barrier;
// the own CTA's with a plain shared store (the warp arrives on the barrier
// after its stores).
__device__ __forceinline__ void send16(bool local, uint32_t addr, uint4 v, uint32_t rbar) {
  if (local)
    st_shared_v4u(addr, v);
  else
    st_async_v4(addr, __uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w), rbar);
}

__device__ __forceinline__ float4 psum4(const float* rb, int C, int rpo, int F, int lr, int f) {  // f % 4 == 0
  float4 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    v[j] = j < C ? *reinterpret_cast<const float4*>(rb + ((size_t)j * rpo + lr) * (F + kRecvPad) + f)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 s = v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j < C) {
      s.x += v[j].x;
      s.y += v[j].y;
      s.z += v[j].z;
      s.w += v[j].w;
    }
  return s;
}
__device__ __forceinline__ float psum(const float* rb, int C, int rpo, int F, int lr, int f) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = j < C ? rb[((size_t)j * rpo + lr) * (F + kRecvPad) + f] : 0.f;
  float s = v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j < C) s += v[j];
  return s;
}

// Constants of the qkv epilogue that do not depend on the frame's data: the
// QK-Norm gains and RoPE cos/sin of this thread's 4 or 8 features.
struct QkvConst {
  float gain[8];
  float c[8], sn[8];
};

__device__ __forceinline__ void load_qkv_const(const KParams& p, const Task& t, int ct, QkvConst& q) {
  const Shape s = shape_of(p);
  const int grp = s.Hq / s.Hkv, w = t.tile % (grp + 2), D = s.D, dpl = D / 16, l16 = ct & 15;
  const uint16_t* gn = (w < grp ? p.q_norm : p.k_norm);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool on = i < dpl && w <= grp;
    q.gain[i] = (on && s.qk_norm) ? bf2f(gn[(size_t)t.layer * D + l16 * dpl + i]) : 1.f;
    const int ip = (l16 & 7) * dpl + i;
    q.c[i] = on ? p.rope[((size_t)t.pos * (D / 2) + ip) * 2] : 1.f;
    q.sn[i] = on ? p.rope[((size_t)t.pos * (D / 2) + ip) * 2 + 1] : 0.f;
  }
}

// x's bf16 operand copy: element (row, f) of position `pos` in the swizzled
// chunk layout the bulk copies of the normed projections read.
__device__ __forceinline__ size_t xb_index(const Shape& s, int pos, int row, int f) {
  const int i = f & 63;
  return (((size_t)pos * (s.H / 64) + (f >> 6)) * s.MR + row) * 64 + ((((i >> 3) ^ (row & 7)) << 3) | (i & 7));
}

// Sums of the C fp16 partials (the normed projections' exchange) in rank
// order, in fp32. Rank j's rows sit at [j * rpo + lr] with a stride of
// F + kRecvPadH halves.
__device__ __forceinline__ float psum_h(const uint16_t* rb, int C, int rpo, int F, int lr, int f) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = j < C ? __half2float(__ushort_as_half(rb[((size_t)j * rpo + lr) * (F + kRecvPadH) + f])) : 0.f;
  float s = v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j < C) s += v[j];
  return s;
}
__device__ __forceinline__ float2 psum2_h(const uint16_t* rb, int C, int rpo, int F, int lr, int f) {  // f even
  float2 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    v[j] = j < C ? __half22float2(*reinterpret_cast<const __half2*>(rb + ((size_t)j * rpo + lr) * (F + kRecvPadH) + f))
                 : make_float2(0.f, 0.f);
  float2 s = v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j < C) { s.x += v[j].x; s.y += v[j].y; }
  return s;
}
__device__ __forceinline__ float4 psum4_h(const uint16_t* rb, int C, int rpo, int F, int lr, int f) {  // f % 4 == 0
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < C) {
      const uint2 u = *reinterpret_cast<const uint2*>(rb + ((size_t)j * rpo + lr) * (F + kRecvPadH) + f);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      if (j == 0) s = make_float4(a.x, a.y, b.x, b.y);
      else { s.x += a.x; s.y += a.y; s.z += b.x; s.w += b.y; }
    }
  }
  return s;
}

// `rb`: the receive slot; fp32 partials for in-proj/o/down, fp16 partials
// already scaled by the norm's row factor for the normed kinds.
// The gains of the RMSNorm that reads x next, for an in-proj/o/down tile's
// output: attention norm of the next layer, MLP norm after o, final norm
// after the last down.
__device__ __forceinline__ const uint16_t* next_gain(const KParams& p, const Shape& s, const Task& t) {
  return t.kind == K_O          ? p.mlp_norm + (size_t)t.layer * s.H
         : t.kind == K_INPROJ   ? p.attn_norm
         : t.layer + 1 < s.L    ? p.attn_norm + (size_t)(t.layer + 1) * s.H
                                : p.final_norm;
}

// `xpre`: in-proj/o/down: [0], [1] this thread's residual values of its first
// two owned rows (o/down; `npre` of them valid), [2] the next norm's gain of
// its feature, all loaded while the MMAs run (`pre_ok`: [2] is valid).
__device__ void epilogue(const KParams& p, const Task& t, const FrameArgs& fa, const float* rb, int C, int rpo,
                         int r0, int nr, int ct, const QkvConst& qc, const float (&xpre)[3], int npre, bool pre_ok) {
  const uint16_t* rh = reinterpret_cast<const uint16_t*>(rb);
  const Shape s = shape_of(p);
  const int F = t.nfeat;
  const int lane = ct & 31, cw = ct >> 5;
  switch (t.kind) {
    case K_INPROJ:
    case K_O:
    case K_DOWN: {  // x (+)= sum; sums of squares per 32 features and x * gain (bf16)
                    // for the norm of x's next reader
      const int nch = s.H / 32;
      const int f = t.tile * 32 + lane;
      const float g = pre_ok ? xpre[2] : bf2f(next_gain(p, s, t)[f]);
      for (int lr = cw, i = 0; lr < nr; lr += 8, ++i) {
        const int row = r0 + lr;
        float* xr = p.x + ((size_t)t.pos * s.MR + row) * s.H + t.tile * 32;
        float v = psum(rb, C, rpo, F, lr, lane);
        if (t.kind != K_INPROJ) v = (i < npre ? (i == 0 ? xpre[0] : xpre[1]) : xr[lane]) + v;
        xr[lane] = v;
        p.xb[xb_index(s, t.pos, row, f)] = f2bf(v * g);
        float q = v * v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
        if (lane == 0) p.ssq[((size_t)t.pos * s.MR + row) * nch + t.tile] = q;
      }
      fence_proxy_async_global();  // x * gain is read by the next projection's bulk copies
      break;
    }
    case K_HEAD: {
      for (int idx = ct; idx < nr * 64; idx += kComputeThreads) {
        const int lr = idx >> 6, f = idx & 63;
        p.logits[((size_t)t.group * s.MR + r0 + lr) * s.V + t.tile * 64 + f] = psum_h(rh, C, rpo, F, lr, f);
      }
      break;
    }
    case K_GU: {  // m = bf16(silu(gate) * up) for the tile's F/2 ffn features, into m's swizzled chunks;
                  // a thread takes 2 consecutive features (one 8-byte partial per rank, one 4-byte store)
      // unrolled by two: at 64 rows each thread takes 3 pairs, and two at a time
      // their partial-sum loads and exponentials overlap (the frame 1 % faster;
      // by three, the larger code gained less)
      const int FF = F / 2, F2 = FF / 2;
#pragma unroll 2
      for (int idx = ct; idx < nr * F2; idx += kComputeThreads) {
        const int lr = idx / F2, i = (idx - lr * F2) * 2, row = r0 + lr;
        const float4 gu = psum4_h(rh, C, rpo, F, lr, 2 * i);  // gate i, up i, gate i+1, up i+1
        const float m0 = gu.x / (1.0f + expf(-gu.x)) * gu.y;
        const float m1 = gu.z / (1.0f + expf(-gu.z)) * gu.w;
        const int fi = t.tile * FF + i, col = fi & 63;  // i even: both features share one 8-element unit
        *reinterpret_cast<uint32_t*>(p.m + ((size_t)(fi >> 6) * s.MR + row) * 64 +
                                     ((((col >> 3) ^ (row & 7)) << 3) | (col & 7))) = pack_bf2(m0, m1);
      }
      fence_proxy_async_global();  // m is read by the down projection's bulk copies
      break;
    }
    case K_QKV: {  // per head: QK-Norm, RoPE, bf16; q to the q buffer, k/v to the frame's KV
      const int grp = s.Hq / s.Hkv;
      const int g = t.tile / (grp + 2), w = t.tile % (grp + 2);
      const int D = s.D, dpl = D / 16;   // 8 or 4 features per thread, 16 threads per row
      const int l16 = ct & 15;
      for (int pass = 0; pass * 16 < nr; ++pass) {
        const int lr = pass * 16 + (ct >> 4);
        const bool valid = lr < nr;
        float v[8];
#pragma unroll
        for (int i4 = 0; i4 < 8; i4 += 4) {
          const float4 a = (i4 < dpl && valid) ? psum4_h(rh, C, rpo, F, lr, l16 * dpl + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i4] = a.x;
          v[i4 + 1] = a.y;
          v[i4 + 2] = a.z;
          v[i4 + 3] = a.w;
        }
        if (w <= grp && s.qk_norm) {
          float q = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) q += v[i] * v[i];
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
          const float sc = rsqrtf(q / (float)D + s.eps);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = v[i] * sc * qc.gain[i];
        }
        if (w <= grp) {  // rotate-half RoPE: pair (i, i + D/2) lives in lanes l16 and l16 ^ 8
          const bool second = l16 >= 8;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, v[i], 8);
            v[i] = second ? v[i] * qc.c[i] + other * qc.sn[i] : v[i] * qc.c[i] - other * qc.sn[i];
          }
        }
        if (valid) {
          const int row = r0 + lr;
          uint16_t* dst;
          if (w < grp) dst = p.q + ((size_t)row * s.Hq + g * grp + w) * D;
          else {
            const int RB = (s.MR + 7) / 8;
            dst = p.kv + (((((size_t)t.layer * s.Hkv + g) * RB + row / 8) * s.P + t.pos) * 8 + (row & 7)) * 2 * D +
                  (w == grp ? 0 : D);
          }
          dst += l16 * dpl;
          if (dpl == 8) {
            uint4 u;
            u.x = pack_bf2(v[0], v[1]); u.y = pack_bf2(v[2], v[3]);
            u.z = pack_bf2(v[4], v[5]); u.w = pack_bf2(v[6], v[7]);
            *reinterpret_cast<uint4*>(dst) = u;
          } else {
            uint2 u;
            u.x = pack_bf2(v[0], v[1]); u.y = pack_bf2(v[2], v[3]);
            *reinterpret_cast<uint2*>(dst) = u;
          }
        }
      }
      fence_proxy_async_global();  // k and v are read by the attention tasks' bulk copies
      break;
    }
  }
}

// The compute leader's share of releasing a task's inputs (see mma_role): after
// tile j's accumulator is complete, the weight pages of that tile the MMA warp
// did not commit, and after the last tile the A slots it did not commit.
// `a0` is the task's first A iteration.
__device__ __forceinline__ void release_inputs(const Task& t, Sm sm, const CState& st, uint32_t a0, int j, int lg) {
  const int nA = 1 << lg;
  const int npages = (t.nkc + t.cpp - 1) / t.cpp, tot_pages = t.ntl * npages;
  for (int pg = 0; pg < npages; ++pg) {
    const int q = j * npages + pg;
    if (q + kNumW >= tot_pages) mb_arrive(sm.bar(B_WEMPTY + (st.w_it + (uint32_t)q) % kNumW));
  }
  if (j == t.ntl - 1)
    for (int c = max(0, t.nkc - nA); c < t.nkc; ++c) mb_arrive(sm.bar(B_AEMPTY + ((a0 + (uint32_t)c) & (nA - 1))));
}

// The partial-sum receive slot of a task's tile number `ri` (counted over the
// CTA's tiles) and the parity of its barriers' phase: an M = 64 handle
// alternates the two slots, an M = 128 one uses both as one slot (its
// two-tile tasks are never planned).
__device__ __forceinline__ int recv_slot(uint32_t ri, bool m128) { return m128 ? 0 : (int)(ri & 1); }
__device__ __forceinline__ uint32_t recv_parity(uint32_t ri, bool m128) { return m128 ? (ri & 1) : ((ri >> 1) & 1); }

__device__ bool proj_task(const KParams& p, const Task& t, const FrameArgs& fa, Sm sm, CState& st, int ct,
                          int gidx, uint32_t tmem) {
  const Shape s = shape_of(p);
  const int R = fa.rows, C = cluster_of(p), F = t.nfeat;
  const int rank = (int)cluster_rank();
  const int rpo = (R + C - 1) / C;
  const int r0 = rank * rpo;
  const int nr = max(0, min(R - r0, rpo));
  const int lane = ct & 31;

  // Before waiting for the predecessor: each tile's rows arriving in its
  // receive slot (no memory traffic; loads wait until after the wait so a
  // late CTA does not spend a round trip on them first).
  const bool normed = t.kind == K_QKV || t.kind == K_GU || t.kind == K_HEAD;
  const int xbytes = normed ? 2 : 4;  // exchange element: fp16 (normed kinds) or fp32
  const bool m128 = m128_of(p);
  if (ct == 0)  // the peers' partials of the owned rows (this CTA's own part is stored locally)
    for (int j = 0; j < t.ntl; ++j)
      mb_expect(sm.bar(B_RFULL + recv_slot(st.recv_it + j, m128)), (uint32_t)((C - 1) * nr * F * xbytes));
  if (!task_wait(p, t, ct, gidx)) return false;

  // 1. activations into the A slots. The normed projections (qkv, gate/up,
  //    heads) read x * gain as bf16 chunks that x's producers wrote; the
  //    norm's per-row factor (mean(x^2) + eps)^(-1/2) multiplies each
  //    partial sum before the exchange (step 2).
  bool ok;
  if (t.kind == K_INPROJ) ok = stage_rows(p, t, fa, sm, st, ct, fa.h, s.T);
  else
    ok = stage_chunks(p, t, fa, sm, st, ct,
                      normed ? p.xb + (size_t)t.pos * s.H * s.MR : (t.kind == K_O ? p.o : p.m));
  // Only the leader's warp can fail inside stage_chunks (its lanes' chunk
  // waits, the leader's refills: the result is made warp-uniform there). All
  // lanes of a warp must take the same branch at the warp-collective waits
  // below, or an abort here would leave the leader in __all_sync and its lanes
  // in wait_bar_w's __syncwarp for good: lane 0 decides for each warp (for the
  // other warps it is true).
  ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
  // With per-chunk waits only the leader's warp has waited so far. o and down
  // read their residual rows below; once one input chunk's producers are done,
  // the phase that last wrote those rows is complete too (a producer tile
  // finishes only after every part of its cluster waited, for its norm's row
  // factor or its own chunks, on the phase before it). This barrier orders the
  // leader's warp's waits before every warp's loads.
  if (t.cbase >= 0 && p.mode == 0 && (t.kind == K_O || t.kind == K_DOWN)) ok = !csync_or(!ok);
  if (ct == 0) trace_stamp(p, gidx, 2);
  // o/down: the residual rows this thread adds to in the epilogue (final since
  // the dependency wait) are loaded now, their latency hidden by the MMAs
  float xpre[3] = {0.f, 0.f, 0.f};
  int npre = 0;
  const bool pre_ok = t.kind == K_INPROJ || t.kind == K_O || t.kind == K_DOWN;
  if (pre_ok) xpre[2] = bf2f(next_gain(p, s, t)[t.tile * 32 + lane]);
  if (t.kind == K_O || t.kind == K_DOWN) {
    const int cw = ct >> 5;
    const float* xt = p.x + ((size_t)t.pos * s.MR + r0) * s.H + t.tile * 32 + lane;
    if (cw < nr) xpre[0] = xt[(size_t)cw * s.H];
    if (cw + 8 < nr) xpre[1] = xt[(size_t)(cw + 8) * s.H];
    npre = 2;
  }
  QkvConst qc;  // epilogue constants: loaded while the MMAs run
  if (t.kind == K_QKV) load_qkv_const(p, t, ct, qc);

  // 2. accumulators -> owners' receive slots, by asynchronous remote stores that
  //    count their bytes on the owner's receive barrier (one slot per tile).
  //    Normed kinds: each sending thread (one row) first computes its row's
  //    norm factor from the per-32-feature sums of squares (fixed order; the
  //    loads overlap the MMAs), scales its partials and sends them as fp16:
  //    the exchange moves half the bytes, and after the row factor the values
  //    are those of a normalized input, far inside the fp16 range (a value
  //    outside it stops the frame with CP_ERR_RANGE).
  const int warp = (ct >> 5) + kComputeBase / 32;
  const int wq = warp & 3, half = (warp - kComputeBase / 32) >> 2;
  // an M = 64 accumulator: warp quadrant wq holds rows 16 wq .. 16 wq + 15 in
  // its first 16 lanes (the other lanes carry no row); M = 128: row 32 wq + lane
  const int row = m128 ? wq * 32 + lane : (lane < 16 ? wq * 16 + lane : kMaxRows);
  const int qrows = m128 ? 32 : 16;
  // The norm's row factor reads the whole row's sums of squares: with
  // per-chunk waits every chunk of x must be done first. Lane i of the
  // leader's warp polls chunk i's counter (by now mostly done: this overlaps
  // the MMAs); the compute barrier publishes it to every warp.
  if (normed && t.cbase >= 0 && p.mode == 0) {
    bool mine = true;
    if (ct < s.H / 64) mine = wait_counter(p, t.cbase + ct, (uint32_t)(t.cpack & 0xFFFF), 0x1400 + t.phase);
    ok = !csync_or(!(ok && mine));
  }
  float srow = 1.f;
  if (normed && row < R) {
    const int nq = s.H / 128;  // float4s of sums of squares per row (<= 16)
    const float4* sp = reinterpret_cast<const float4*>(p.ssq + ((size_t)t.pos * s.MR + row) * (s.H / 32));
    float sum = 0.f;
    for (int hb = 0; hb < nq; hb += 8) {
      float4 sq[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) sq[c] = hb + c < nq ? sp[hb + c] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        sum += sq[c].x;
        sum += sq[c].y;
        sum += sq[c].z;
        sum += sq[c].w;
      }
    }
    srow = rsqrtf(sum / (float)s.H + s.eps);
  }
  for (int j = 0; j < t.ntl; ++j) {
    const uint32_t ai = st.acc_it + j, ri = st.recv_it + j;
    const int acc = ai % kNumAcc, b = recv_slot(ri, m128);
    if (ok) ok = wait_bar_w(p, sm.bar(B_ACCFULL + acc), (ai / kNumAcc) & 1, 0x3000);
    if (ct == 0 && ok) release_inputs(t, sm, st, st.a_it - (uint32_t)t.nkc, j, a_log2(p));
    if (ok) ok = wait_bar_w(p, sm.bar(B_RFREE + b), recv_parity(ri, m128) ^ 1, 0x3100, true);
    ok = __all_sync(0xffffffffu, ok);
    if (ct == 0 && j == 0) trace_stamp(p, gidx, 3);
    if (ok && wq * qrows < R) {
      tm_fence_after();
      const int cb = half * (F / 2);
      const int owner = row < R ? row / rpo : 0, lr = row - owner * rpo;
      const bool local = owner == rank;  // own rows: plain shared stores, no cluster traffic
      const uint32_t rbar = mapa(sm.bar(B_RFULL + b), (uint32_t)owner);
      const uint32_t tbase = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * kAccCols + cb);
      if (normed) {  // fp16 after the row factor; F / 2 is a multiple of 32 (64 or 32 features per half)
        const uint32_t offh = (uint32_t)(((rank * rpo + lr) * (F + kRecvPadH) + cb) * 2);
        const uint32_t dsth = local ? sm.recv(b) + offh : mapa(sm.recv(b) + offh, (uint32_t)owner);
        bool range_ok = true;
#pragma unroll 1
        for (int cc = 0; cc < F / 2; cc += 32) {
          float v[32];
          tm_ld32(tbase + cc, v);
          uint32_t h2[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float a = v[2 * q] * srow, c = v[2 * q + 1] * srow;
            range_ok = range_ok && fabsf(a) <= 65504.f && fabsf(c) <= 65504.f;
            const __half2 hv = __floats2half2_rn(a, c);
            h2[q] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          if (row < R) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              send16(local, dsth + (cc + 8 * q) * 2, make_uint4(h2[4 * q], h2[4 * q + 1], h2[4 * q + 2], h2[4 * q + 3]),
                     rbar);
          }
        }
        if (row < R && !range_ok) raise_error(p, CP_ERR_RANGE, 0x3400 + t.kind);
      } else if ((F / 2) % 32 == 0) {
        const uint32_t off = (uint32_t)(((rank * rpo + lr) * (F + kRecvPad) + cb) * 4);
        const uint32_t dst = local ? sm.recv(b) + off : mapa(sm.recv(b) + off, (uint32_t)owner);
#pragma unroll 1
        for (int cc = 0; cc < F / 2; cc += 32) {
          float v[32];
          tm_ld32(tbase + cc, v);
          if (row < R) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              send16(local, dst + (cc + 4 * q) * 4,
                     make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                                __float_as_uint(v[4 * q + 3])),
                     rbar);
          }
        }
      } else {
        const uint32_t off = (uint32_t)(((rank * rpo + lr) * (F + kRecvPad) + cb) * 4);
        const uint32_t dst = local ? sm.recv(b) + off : mapa(sm.recv(b) + off, (uint32_t)owner);
#pragma unroll 1
        for (int cc = 0; cc < F / 2; cc += 16) {
          float v[16];
          tm_ld16(tbase + cc, v);
          if (row < R) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              send16(local, dst + (cc + 4 * q) * 4,
                     make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                                __float_as_uint(v[4 * q + 3])),
                     rbar);
          }
        }
      }
    }
    tm_fence_before();
    __syncwarp();
    if (lane == 0 && ok) {
      mb_arrive(sm.bar(B_ACCEMPTY + acc));
      mb_arrive(sm.bar(B_RFULL + b));  // this warp's stores of the own rows (release, CTA scope)
    }
  }
  st.acc_it += t.ntl;
  st.w_it += (uint32_t)(t.ntl * ((t.nkc + t.cpp - 1) / t.cpp));

  // 3. own rows: add the C partials in rank order, epilogue, store
  for (int j = 0; j < t.ntl; ++j) {
    const uint32_t ri = st.recv_it + j;
    if (ok) ok = wait_bar_w(p, sm.bar(B_RFULL + recv_slot(ri, m128)), recv_parity(ri, m128), 0x3200, true);
    if (ct == 0 && j == 0) trace_stamp(p, gidx, 4);
    if (ok) {
      if (j == 0) {
        epilogue(p, t, fa, sm.recv_ptr(recv_slot(ri, m128)), C, rpo, r0, nr, ct, qc, xpre, npre, pre_ok);
      } else {
        Task tj = t;
        tj.tile = t.tile + j;
        if (t.kind == K_QKV) load_qkv_const(p, tj, ct, qc);
        epilogue(p, tj, fa, sm.recv_ptr(recv_slot(ri, m128)), C, rpo, r0, nr, ct, qc, xpre, 0, false);
      }
    }
  }
  const uint32_t r_first = st.recv_it;
  st.recv_it += t.ntl;
  if (!finish_and_signal(p, t, ct, gidx, ok)) return false;
  if (ct == 0 && t.ntl == 2 && p.mode == 0) {  // the second tile's counter (its kv group's for qkv)
    red_release_add(p.counters + t.signal_b, 1);
  }
  // Free the receive slots on every CTA of the cluster, one lane per CTA. The
  // arrive only has to follow this CTA's reads of the slots, and those were
  // all performed before the compute warps' barrier in finish_and_signal, so
  // it is relaxed: with release semantics it also waited for the signal's
  // release-add to reach global memory (about 1 us per task, measured).
  if (ct < C)
    for (int j = 0; j < t.ntl; ++j)
      mb_arrive_cluster_relaxed(mapa(sm.bar(B_RFREE + recv_slot(r_first + j, m128)), (uint32_t)ct));
  return true;
}

// ---------------------------------------------------------------- attention
// Warp-level attention of one row over positions 0..pos for the G q heads of
// one kv group, from the keys and values staged in shared memory ([position]
// [row][key|value][D]). Each key and value load serves all G heads, and the G
// heads' shuffle trees are independent, so they interleave.
template <int G>
__device__ __forceinline__ void attn_rows(const KParams& p, Sm sm, const uint2 (&qraw)[4], int cw, int lane, int row,
                                          int g, int pos) {
  const Shape s = shape_of(p);
  const int D = s.D, dpl = D / 32;
  const uint8_t* kvb = sm.base + kSmemA + (size_t)cw * 2 * D * 2 + lane * dpl * 2;  // + tt * tstride
  const size_t tstride = (size_t)8 * 2 * D * 2;
  const int mytt = lane & 15;
  float q[G][4];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    q[hh][0] = __uint_as_float(qraw[hh].x << 16);
    q[hh][1] = __uint_as_float(qraw[hh].x & 0xFFFF0000u);
    q[hh][2] = __uint_as_float(qraw[hh].y << 16);
    q[hh][3] = __uint_as_float(qraw[hh].y & 0xFFFF0000u);
  }
  float pd[G][16];
#pragma unroll
  for (int tt = 0; tt < 16; ++tt) {  // positions past pos read stale scratch: selected away
    float k[4];
    if (dpl == 4) {
      const uint2 kk = *reinterpret_cast<const uint2*>(kvb + tt * tstride);
      k[0] = __uint_as_float(kk.x << 16); k[1] = __uint_as_float(kk.x & 0xFFFF0000u);
      k[2] = __uint_as_float(kk.y << 16); k[3] = __uint_as_float(kk.y & 0xFFFF0000u);
    } else {
      const uint32_t kk = *reinterpret_cast<const uint32_t*>(kvb + tt * tstride);
      k[0] = __uint_as_float(kk << 16); k[1] = __uint_as_float(kk & 0xFFFF0000u);
      k[2] = k[3] = 0.f;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float d = q[hh][0] * k[0] + q[hh][1] * k[1] + q[hh][2] * k[2] + q[hh][3] * k[3];
      pd[hh][tt] = tt <= pos ? d : 0.f;
    }
  }
  // reduce-scatter: after the step with offset o, the lane keeps the half of
  // its positions whose bit log2(o) equals its own lane bit
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int jj = 0; jj < o; ++jj) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float keep = hi ? pd[hh][o + jj] : pd[hh][jj];
        const float give = hi ? pd[hh][jj] : pd[hh][o + jj];
        pd[hh][jj] = keep + __shfl_xor_sync(0xffffffffu, give, o);
      }
    }
  }
  float w[G], z[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const float dot = pd[hh][0] + __shfl_xor_sync(0xffffffffu, pd[hh][0], 16);
    const float sc = mytt <= pos ? dot * p.attn_scale : -INFINITY;
    float mx = sc;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    w[hh] = mytt <= pos ? expf(sc - mx) : 0.f;
    z[hh] = w[hh];
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) z[hh] += __shfl_xor_sync(0xffffffffu, z[hh], o);
  }
  float acc[G][4];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.f;
  // positions 0..pos only, rolled up: nothing here indexes a register array by
  // the position, and a smaller loop body keeps the kernel's code footprint down
  // (measured faster than the 16 predicated iterations)
#pragma unroll 1
  for (int tt = 0; tt <= pos; ++tt) {
    float v[4];
    const uint8_t* vp = kvb + tt * tstride + D * 2;
    if (dpl == 4) {
      const uint2 vv = *reinterpret_cast<const uint2*>(vp);
      v[0] = __uint_as_float(vv.x << 16); v[1] = __uint_as_float(vv.x & 0xFFFF0000u);
      v[2] = __uint_as_float(vv.y << 16); v[3] = __uint_as_float(vv.y & 0xFFFF0000u);
    } else {
      const uint32_t vv = *reinterpret_cast<const uint32_t*>(vp);
      v[0] = __uint_as_float(vv << 16); v[1] = __uint_as_float(vv & 0xFFFF0000u);
      v[2] = v[3] = 0.f;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float wt = __shfl_sync(0xffffffffu, w[hh], tt);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[hh][e] += wt * v[e];
    }
  }
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    // o feature f = h*D + lane*dpl + i -> chunk f/64, unit (f%64)/8 swizzled by row
    const int f0 = (g * G + hh) * D + lane * dpl;
    const int chunk = f0 >> 6, col = f0 & 63;
    uint16_t* dst = p.o + ((size_t)chunk * s.MR + row) * 64 + ((((col >> 3) ^ (row & 7)) << 3) | (col & 7));
    if (dpl == 4) {
      uint2 u;
      u.x = pack_bf2(acc[hh][0] / z[hh], acc[hh][1] / z[hh]);
      u.y = pack_bf2(acc[hh][2] / z[hh], acc[hh][3] / z[hh]);
      *reinterpret_cast<uint2*>(dst) = u;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf2(acc[hh][0] / z[hh], acc[hh][1] / z[hh]);
    }
  }
}

// One kv group x one block of 8 rows at position pos. The block's keys and
// values for positions 0..pos are one contiguous region of the cache
// ([position][row][key|value][D]); the leader brings it into the scratch area
// (the A slots, idle between projections) with one bulk copy. Warp w takes
// row 8*block + w and every q head of the group. The lanes split D for the
// partial dot products of all 16 positions; a reduce-scatter over the lanes
// (xor 8, 4, 2, 1, then 16: a fixed tree) leaves lane L with the score of
// position L mod 16, so the softmax is one exp per lane and two 4-step
// trees. The value sum in fp32 broadcasts each weight from its lane; the
// output is rounded to bf16 into the swizzled chunks the o projection streams.
static_assert(kRowBlock == 8 && kMaxPositions == 16, "attention lane mapping");
static_assert(kMaxPositions * kRowBlock * 2 * 128 * 2 <= kNumA * kAChunkBytes, "attention scratch");
__device__ bool attn_task(const KParams& p, const Task& t, const FrameArgs& fa, Sm sm, CState& st, int ct, int gidx) {
  const Shape s = shape_of(p);
  const int R = fa.rows, grp = s.Hq / s.Hkv, D = s.D, dpl = D / 32;
  const int lane = ct & 31, cw = ct >> 5, g = t.group, pos = t.pos;
  const int r0 = t.tile * kRowBlock;
  const int nrows = min(kRowBlock, R - r0);
  const int row = r0 + cw;
  const bool live = cw < nrows;
  // The row block's keys and values of positions 0..pos are one contiguous
  // region. Positions before pos were written by earlier positions' qkv
  // phases: thread 32 (its own warp, so the poll runs beside the leader's
  // dependency wait) checks the group's previous-position counter, which is
  // long complete, and copies them before this task's own dependency is met;
  // only position pos's 4 KB follow it, issued by the leader. The early copy
  // only raises the barrier's byte count; the arrival comes with the last
  // copy, so the phase completes once every byte has landed. The compute
  // barrier in task_wait orders thread 32's byte count and flag before the
  // leader's arrival.
  const uint32_t bar = sm.bar(B_SCR);
  const int RB = (s.MR + 7) / 8;
  const size_t off = ((((size_t)t.layer * s.Hkv + g) * RB + t.tile) * s.P) * 8 * 2 * D;
  const uint32_t per = 8 * 2 * D * 2;  // one position's keys and values of the row block
  volatile uint32_t* eflag = sm.misc_u32(kMiscEarly);
  if (ct == 32) {
    uint32_t e = 0;
    if (nrows > 0 && pos > 0 && p.mode == 0 && t.wait1 >= 0 &&
        wait_counter(p, t.wait1, (uint32_t)t.target1, 0x1800)) {
      fence_proxy_async_global();
      mb_expect_tx(bar, (uint32_t)pos * per);
      bulk_g2s(sm.a_slot(0), p.kv + off, (uint32_t)pos * per, bar);
      e = 1;
    }
    *eflag = e;
  }
  if (!task_wait(p, t, ct, gidx)) {
    if (ct == 0 && *eflag) {  // the early copy's phase completes; the teardown drain waits for it
      mb_arrive(bar);
      st.scr_it++;
    }
    return false;
  }
  if (nrows > 0 && ct == 0) {
    const uint32_t first = *eflag ? (uint32_t)pos : 0u;
    fence_proxy_async_global();
    mb_expect(bar, ((uint32_t)pos + 1 - first) * per);
    bulk_g2s(sm.a_slot(0) + first * per, p.kv + off + (size_t)first * (per / 2), ((uint32_t)pos + 1 - first) * per, bar);
  }
  // this warp's q (dpl values of each head of the group), loaded before the copy lands
  uint2 qraw[4];
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    qraw[hh] = make_uint2(0u, 0u);
    if (live && hh < grp) {
      const uint16_t* qp = p.q + ((size_t)row * s.Hq + g * grp + hh) * D + lane * dpl;
      qraw[hh] = dpl == 4 ? *reinterpret_cast<const uint2*>(qp) : make_uint2(*reinterpret_cast<const uint32_t*>(qp), 0u);
    }
  }
  bool ok = true;
  if (nrows > 0) {
    const uint32_t it = st.scr_it++;
    ok = wait_bar_w(p, sm.bar(B_SCR), it & 1, 0x2200);
  }
  if (ok && live) {
    switch (grp) {
      case 1: attn_rows<1>(p, sm, qraw, cw, lane, row, g, pos); break;
      case 2: attn_rows<2>(p, sm, qraw, cw, lane, row, g, pos); break;
      default: attn_rows<4>(p, sm, qraw, cw, lane, row, g, pos); break;
    }
  }
  fence_proxy_async_global();  // o is read by the o projection's bulk copies
  return finish_and_signal(p, t, ct, gidx, ok);
}

// ---------------------------------------------------------------- draw
// Block-wide helpers over the 256 compute threads; `red` is shared scratch of
// at least 8 words per call site. Results are identical in every thread and
// every reduction runs in a fixed order.
__device__ __forceinline__ uint32_t f_ord(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block reductions over the 256 compute threads: a warp tree, each warp's
// result (lane 0's) in shared memory, one barrier, then every thread combines
// the 8 in warp order. Two buffers alternate, so one barrier per reduction
// suffices: a buffer is written again only after the next reduction's
// barrier, which every thread reaches after reading it.
struct DrawRed {
  uint32_t* buf;  // [2][8 warps][4 words]
  int k;          // reductions so far
  __device__ uint32_t* next() { return buf + (k++ & 1) * 32; }
};

__device__ __forceinline__ void better(float& v, int& i, uint32_t& key, float ov, int oi, uint32_t ok) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; key = ok; }
}

// Largest value, lowest index on ties (a total order: every thread ends with
// the same winner), carrying the winner's key.
__device__ __forceinline__ void red_argmax(DrawRed& r, int ct, float& v, int& i, uint32_t& key) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    const uint32_t ok = __shfl_xor_sync(0xffffffffu, key, o);
    better(v, i, key, ov, oi, ok);
  }
  uint32_t* b = r.next();
  if ((ct & 31) == 0) {
    b[(ct >> 5) * 4] = __float_as_uint(v);
    b[(ct >> 5) * 4 + 1] = (uint32_t)i;
    b[(ct >> 5) * 4 + 2] = key;
  }
  csync();
  v = __uint_as_float(b[0]);
  i = (int)b[1];
  key = b[2];
  for (int w = 1; w < 8; ++w) better(v, i, key, __uint_as_float(b[w * 4]), (int)b[w * 4 + 1], b[w * 4 + 2]);
}

// A float sum and an int count together (lane 0's tree order, then warps in order).
__device__ __forceinline__ void red_sum2(DrawRed& r, int ct, float& a, int& c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
  }
  uint32_t* b = r.next();
  if ((ct & 31) == 0) {
    b[(ct >> 5) * 4] = __float_as_uint(a);
    b[(ct >> 5) * 4 + 1] = (uint32_t)c;
  }
  csync();
  a = __uint_as_float(b[0]);
  c = (int)b[1];
  for (int w = 1; w < 8; ++w) {
    a += __uint_as_float(b[w * 4]);
    c += (int)b[w * 4 + 1];
  }
}

constexpr int kVpt = kMaxVocab / kComputeThreads;  // logits per thread (8)
constexpr int kDrawHist = 512;                       // after the reduction buffers: 4 histograms
constexpr int kDrawGumbel = kDrawHist + 4 * 256 * 4; // then the row's Gumbel noise (V floats)
constexpr int kDrawScratch = kDrawGumbel + kMaxVocab * 4;
static_assert(kDrawScratch <= kNumA * kAChunkBytes, "the draw's scratch fits the A slots it borrows");

// The Gumbel noise -log(-log(u)) of every token of one row, u from Philox4x32-10
// with key = seed and counter = (v / 4, row, offset): token v takes word v % 4
// of counter v / 4. It does not depend on the logits, so it is made (threads
// t0, t0 + nt, ... taking one counter each) before the draw's dependency is
// met; `g` is the draw scratch's noise area.
__device__ __forceinline__ void gumbel_fill(float* g, int V, uint64_t seed, int row, int64_t off, int t0, int nt) {
  const uint2 k2 = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t olo = (uint32_t)(uint64_t)off, ohi = (uint32_t)((uint64_t)off >> 32);
#pragma unroll 1
  for (int m = t0; m < V / 4; m += nt) {
    const uint4 w = philox10(make_uint4((uint32_t)m, (uint32_t)row, olo, ohi), k2);
    float4 r;
    r.x = -logf(-logf(philox_uniform(w.x)));
    r.y = -logf(-logf(philox_uniform(w.y)));
    r.z = -logf(-logf(philox_uniform(w.z)));
    r.w = -logf(-logf(philox_uniform(w.w)));
    reinterpret_cast<float4*>(g)[m] = r;
  }
}
// The radix select's histograms start at zero: zeroed before the barrier that
// precedes the draw (the dependency wait's, in the frame).
__device__ __forceinline__ void draw_zero_hist(uint8_t* scratch, int ct) {
  int* hist = reinterpret_cast<int*>(scratch + kDrawHist);
#pragma unroll
  for (int q = 0; q < 4; ++q) hist[q * 256 + ct] = 0;
}

// One row's draw on the 256 compute threads. Thread ct holds entries
// ct*vpt .. ct*vpt+vpt-1. Scratch: kDrawScratch bytes of shared memory, its
// histograms zeroed (draw_zero_hist) and its noise made (gumbel_fill) before a
// compute barrier that precedes the call.
//  * top-k: the k-th largest key by most-significant-digit radix select (up
//    to 4 passes of 8 bits, each with its own histogram, zeroed up front;
//    after a pass's barrier every warp scans the histogram itself, so a pass
//    costs one barrier; it stops once the selected bin is kept whole), ties
//    on that key kept by lowest index;
//  * top-p: softmax over the kept set; the Gumbel-max candidate is accepted
//    when the mass of kept tokens ranked above it is below p (the first token
//    always is), else dropped and the next best tried.
// `emb` (optional): the embedding table the drawn code indexes (rows of `H`
// bf16); the first candidate's row is prefetched into L2 while top-p checks it.
__device__ __forceinline__ int draw_row(const float* lg_row, int V, float T, int topk, float topp, uint8_t* scratch,
                                     int ct, const uint16_t* emb = nullptr, int H = 0) {
  const int vpt = V / kComputeThreads, lane = ct & 31;
  DrawRed red{reinterpret_cast<uint32_t*>(scratch), 0};
  int* hist = reinterpret_cast<int*>(scratch + kDrawHist);   // [4][256]
  const float* gum = reinterpret_cast<const float*>(scratch + kDrawGumbel);
  float lg[kVpt];
  if (vpt == kVpt) {  // two 16-byte loads per thread
    const float4* l4 = reinterpret_cast<const float4*>(lg_row) + ct * 2;
    const float4 a = l4[0], b = l4[1];
    lg[0] = a.x; lg[1] = a.y; lg[2] = a.z; lg[3] = a.w;
    lg[4] = b.x; lg[5] = b.y; lg[6] = b.z; lg[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < kVpt; ++i) lg[i] = i < vpt ? lg_row[ct * vpt + i] : -INFINITY;
  }

  if (!(T > 0.f)) {  // greedy: largest logit, lowest index on ties
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    uint32_t bk = 0;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
      if (i < vpt) better(bv, bi, bk, lg[i], ct * vpt + i, 0u);
    red_argmax(red, ct, bv, bi, bk);
    return bi;
  }
  float sv[kVpt];
  uint32_t key[kVpt];
#pragma unroll
  for (int i = 0; i < kVpt; ++i) {
    sv[i] = i < vpt ? lg[i] / T : -INFINITY;
    key[i] = i < vpt ? f_ord(sv[i]) : 0u;
  }
  const bool use_k = topk >= 1 && topk < V;
  const bool use_p = topp < 1.0f;
  // the largest score (always kept: the softmax reference of top-p) rides on
  // the first radix pass's barrier (its own, without top-k)
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kVpt; ++i) mx = fmaxf(mx, sv[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  uint32_t* mxb = red.next();
  if (lane == 0) mxb[(ct >> 5) * 4] = __float_as_uint(mx);
  if (!use_k) csync();
  uint32_t kth = 0;
  int need = 0, n_eq = 0;
  if (use_k) {
    uint32_t prefix = 0;
    need = topk;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
      int* h = hist + pass * 256;
#pragma unroll
      for (int i = 0; i < kVpt; ++i)
        if (i < vpt && (key[i] & hmask) == prefix) atomicAdd(&h[(key[i] >> shift) & 255u], 1);
      csync();
      // every warp finds the bin holding the need-th largest, scanning from the top
      int b[8], ls = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { b[i] = h[lane * 8 + i]; ls += b[i]; }
      int incl = ls;  // sum over lanes >= this lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      const int above = incl - ls;  // lanes > this lane
      const bool own = above < need && incl >= need;  // exactly one lane
      int bin = 0, nneed = 0, neq = 0;
      if (own) {
        int acc = above;
        for (int i = 7; i >= 0; --i) {
          if (acc + b[i] >= need) {
            bin = lane * 8 + i;
            nneed = need - acc;
            neq = b[i];
            break;
          }
          acc += b[i];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, own)) - 1;
      bin = __shfl_sync(0xffffffffu, bin, src);
      nneed = __shfl_sync(0xffffffffu, nneed, src);
      neq = __shfl_sync(0xffffffffu, neq, src);
      prefix |= (uint32_t)bin << shift;
      need = nneed;
      n_eq = neq;
      // every key of the bin is needed: the kept set is the bin and all above
      // it, whatever the lower digits (usually after two passes), so the
      // threshold stops at the bin's smallest key and keeps all its ties
      if (nneed == neq) {
        need = V;
        n_eq = V;
        break;
      }
    }
    kth = prefix;
  }
  mx = __uint_as_float(mxb[0]);
  for (int w = 1; w < 8; ++w) mx = fmaxf(mx, __uint_as_float(mxb[w * 4]));
  bool keep[kVpt];
  {
    int eq_before = 0;
    if (use_k && need < n_eq) {  // ties on the threshold key: rank them by index
      int mine = 0;
#pragma unroll
      for (int i = 0; i < kVpt; ++i) mine += (i < vpt && key[i] == kth) ? 1 : 0;
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t* b = red.next();
      if (lane == 31) b[(ct >> 5) * 4] = (uint32_t)incl;
      csync();
      int wbase = 0;
      for (int w = 0; w < (ct >> 5); ++w) wbase += (int)b[w * 4];
      eq_before = wbase + incl - mine;
    }
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
      bool k_ok = i < vpt;
      if (use_k && k_ok) {
        if (key[i] > kth) k_ok = true;
        else if (key[i] == kth) { k_ok = eq_before < need; eq_before++; }
        else k_ok = false;
      }
      keep[i] = k_ok;
    }
  }
  // softmax weights of the kept set relative to the largest score (needed by top-p)
  float e[kVpt];
  float Z = 1.f;
  if (use_p) {
    float z = 0.f;
    int unused = 0;
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
      e[i] = keep[i] ? expf(sv[i] - mx) : 0.f;
      z += e[i];
    }
    red_sum2(red, ct, z, unused);
    Z = z;
  }
  // Gumbel-perturbed scores (the noise was made before the dependency)
  float z[kVpt];
#pragma unroll
  for (int i = 0; i < kVpt; ++i) z[i] = (i < vpt && keep[i]) ? sv[i] + gum[ct * vpt + i] : -INFINITY;
  // best perturbed score among the kept; with top-p, accept it only if the
  // softmax mass of kept tokens ranked above it is below top_p (the first
  // token is always kept), else drop it and try the next
  for (int iter = 0; iter < V; ++iter) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    uint32_t bk = 0;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
      if (i < vpt && z[i] > -INFINITY) better(bv, bi, bk, z[i], ct * vpt + i, key[i]);
    red_argmax(red, ct, bv, bi, bk);
    if (bi == 0x7fffffff) return 0;  // cannot happen: the first kept token is always accepted
    if (iter == 0 && emb && ct * 64 < H) prefetch_l2(emb + (size_t)bi * H + ct * 64);
    if (!use_p) return bi;
    float ma = 0.f;
    int ca = 0;
#pragma unroll
    for (int i = 0; i < kVpt; ++i) {
      const int v = ct * vpt + i;
      if (keep[i] && (key[i] > bk || (key[i] == bk && v < bi))) { ma += e[i]; ca += 1; }
    }
    red_sum2(red, ct, ma, ca);
    if (ca == 0 || ma / Z < topp) return bi;
#pragma unroll
    for (int i = 0; i < kVpt; ++i)
      if (i < vpt && ct * vpt + i == bi) z[i] = -INFINITY;
  }
  return 0;
}

// Write table `tab`'s embedding of `code` as position `xpos`'s input (if
// xpos < P) with its per-32-feature sums of squares, and add it to (or start)
// the row's embedding sum.
__device__ __forceinline__ void embed_row(const KParams& p, float* emb_sum, int tab, int code, int row, int xpos, bool first,
                                       int ct) {
  // Warp cw takes 32-feature chunks cw, cw+8, ... (H <= 2048: at most 8);
  // every load is issued before the first store, one round trip in all.
  const Shape s = shape_of(p);
  const uint16_t* e = p.embed + ((size_t)tab * s.V + code) * s.H;
  const int lane = ct & 31, cw = ct >> 5, nch = s.H / 32;
  float* xr = xpos < s.P ? p.x + ((size_t)xpos * s.MR + row) * s.H : nullptr;
  float* es = emb_sum + (size_t)row * s.H;
  float v[8], g[8], old[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = cw + 8 * k, f = c * 32 + lane;
    v[k] = g[k] = old[k] = 0.f;
    if (c < nch) {
      v[k] = bf2f(e[f]);
      if (xr) g[k] = bf2f(p.attn_norm[f]);
      if (!first) old[k] = es[f];
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = cw + 8 * k, f = c * 32 + lane;
    if (c < nch) {
      if (xr) {
        xr[f] = v[k];
        p.xb[xb_index(s, xpos, row, f)] = f2bf(v[k] * g[k]);
        float q = v[k] * v[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
        if (lane == 0) p.ssq[((size_t)xpos * s.MR + row) * nch + c] = q;
      }
      es[f] = first ? v[k] : old[k] + v[k];
    }
  }
  if (xr) fence_proxy_async_global();  // x * gain is read by the first qkv projection's bulk copies
}

// Task and frame arguments come by value, so their fields stay in registers.
// The draw path is inlined like the waits (no register save and restore
// through local memory at each call: measured 1.7 % faster).
__device__ __forceinline__ bool draw_task(const KParams& p, const Task t, const FrameArgs fa, Sm sm, int ct, int gidx) {
  const Shape s = shape_of(p);
  const int row = t.tile, j = t.group;
  const bool live = row < fa.rows;
  // the row's embedding sum and the next norm's gains do not depend on the
  // draw: their lines are on their way to L2 while the draw runs (not from
  // the leader, whose dependency poll would queue behind its requests)
  if (live) {
    if (ct >= 32 && (ct - 32) * 32 < s.H) prefetch_l2(fa.emb_sum + (size_t)row * s.H + (ct - 32) * 32);
    else if (ct >= 160 && (ct - 160) * 64 < s.H) prefetch_l2(p.attn_norm + (ct - 160) * 64);
  }
  // the noise and the zeroed histograms, published by the dependency wait's
  // barrier: the six compute warps that share no scheduler with the polling
  // leader (compute warps 0 and 4 sit on the same one) make the noise while
  // it polls (the offset is written only by the row's last draw, after its
  // own read)
  draw_zero_hist(sm.scratch(), ct);
  if (live && ct >= 32 && (ct >> 5) != 4)
    gumbel_fill(reinterpret_cast<float*>(sm.scratch() + kDrawGumbel), s.V, fa.seed[row], row, fa.offset[row] + j,
                ct < 128 ? ct - 32 : ct - 64, kComputeThreads - 64);
  if (!task_wait(p, t, ct, gidx)) return false;
  // the row's sampler settings: read after the wait (their latency overlaps
  // the logits'), so nothing is queued ahead of the leader's poll
  float T = 0.f, tp = 1.f;
  int tk = 0;
  int64_t base = 0;
  if (live) {
    T = fa.temperature[row];
    tk = fa.top_k[row];
    tp = fa.top_p[row];
    if (ct == 0 && j == s.P - 2) base = fa.offset[row];
  }
  if (live) {
    int code = draw_row(p.logits + ((size_t)j * s.MR + row) * s.V, s.V, T, tk, tp, sm.scratch(), ct,
                        p.embed + (size_t)(j + 1) * s.V * s.H, s.H);
    if (code < 0 || code >= s.V) {  // cannot happen; never index out of the table
      if (ct == 0) raise_error(p, CP_ERR_DEVICE_BOUNDS, 0x5000 + j);
      code = 0;
    }
    if (ct == 0) {
      fa.codes[(size_t)row * (s.P - 1) + j] = code;
      if (j == s.P - 2) fa.offset[row] = base + (s.P - 1);
    }
    embed_row(p, fa.emb_sum, j + 1, code, row, t.pos, false, ct);
  }
  return finish_and_signal(p, t, ct, gidx, true);
}

__device__ __forceinline__ bool emb0_task(const KParams& p, const Task t, const FrameArgs fa, int ct, int gidx) {
  if (!task_wait(p, t, ct, gidx)) return false;
  const int row = t.tile;
  if (row < fa.rows) {
    int code = fa.c0[row];
    if (code < 0 || code >= shape_of(p).V) {
      if (ct == 0) raise_error(p, CP_ERR_DEVICE_BOUNDS, 0x5100);
      code = 0;
    }
    embed_row(p, fa.emb_sum, 0, code, row, 1, true, ct);
  }
  return finish_and_signal(p, t, ct, gidx, true);
}

// ---------------------------------------------------------------- roles
__device__ void producer_role(const KParams& p, const Task* tl, int n, int gbase, Sm sm, uint32_t& w_it) {
  const uint64_t pol = policy_evict_first();
  Task nxt;
  if (n > 0) nxt = tl[0];
  for (int i = 0; i < n; ++i) {
    const Task t = nxt;  // register copy; the next record's load is in flight during this task
    if (i + 1 < n) nxt = tl[i + 1];
    if (t.type != T_PROJ) continue;
    const int npages = (t.nkc + t.cpp - 1) / t.cpp;
    const uint32_t chunk_bytes = (uint32_t)t.nfeat * 128u;
    const size_t unit = (size_t)t.nkc * chunk_bytes;
    for (int j = 0; j < t.ntl; ++j) {  // tile j's part sits C parts after tile j-1's
      const uint8_t* src = p.wpack + t.w_off + (size_t)j * cluster_of(p) * unit;
      for (int pg = 0; pg < npages; ++pg) {
        const int slot = w_it % kNumW;
        if (!wait_bar(p, sm.bar(B_WEMPTY + slot), ((w_it / kNumW) & 1) ^ 1, 0x4000, false, true)) return;
        const int nch = min(t.cpp, t.nkc - pg * t.cpp);
        const uint32_t bytes = (uint32_t)nch * chunk_bytes;
        mb_expect(sm.bar(B_WFULL + slot), bytes);
        bulk_g2s_hint(sm.w_page(slot), src + (size_t)pg * t.cpp * chunk_bytes, bytes, sm.bar(B_WFULL + slot), pol);
        w_it++;
      }
    }
    trace_stamp(p, gbase + i, 11);
  }
}

// Tile j of a task accumulates into TMEM buffer (acc_it + j) % kNumAcc. The loop is
// kept lean (page-major, no division by a runtime value, one A wait per chunk
// for the task's first tile only): its per-chunk overhead sits on the critical
// path of every projection phase. A commit costs about as much as an MMA
// issue, so the MMA warp commits only the accumulator, plus the A slots and
// weight pages the task itself needs again (a chunk c with c + kNumA < nkc, a
// page q of the task's ntl * npages with q + kNumW < ntl * npages); the compute
// leader releases the rest with plain arrivals once it has seen the
// accumulator (release_inputs). Every tile reads the same staged K part.
__device__ void mma_role(const KParams& p, const Task* tl, int n, int gbase, Sm sm, uint32_t tmem) {
  uint32_t w_it = 0, a_it = 0, acc_it = 0;
  Task nxt;
  if (n > 0) nxt = tl[0];
  for (int i = 0; i < n; ++i) {
    const Task t = nxt;  // register copy; the next record's load is in flight during this task
    if (i + 1 < n) nxt = tl[i + 1];
    if (t.type != T_PROJ) continue;
    // M = 64: the A slots hold 64 rows and no rows beyond them are read;
    // M = 128: a chunk is two adjacent slots
    const bool m128 = m128_of(p);
    const int lg = a_log2(p), nA = 1 << lg;
    const uint32_t idesc = m128 ? idesc_bf16_m128(t.nfeat) : idesc_bf16_m64(t.nfeat);
    const uint32_t chunk_bytes = (uint32_t)t.nfeat * 128u;
    const int nkc = t.nkc, cpp = t.cpp, npages = (nkc + cpp - 1) / cpp, tot_pages = t.ntl * npages;
    for (int j = 0; j < t.ntl; ++j) {
      const int acc = acc_it % kNumAcc;
      if (!wait_bar(p, sm.bar(B_ACCEMPTY + acc), ((acc_it / kNumAcc) & 1) ^ 1, 0x4100)) return;
      if (j == 0) trace_stamp(p, gbase + i, 8);
      tm_fence_after();
      const uint32_t d = tmem + (uint32_t)(acc * kAccCols);
      const bool last = j == t.ntl - 1;
      int kc = 0;
      for (int pg = 0; pg < npages; ++pg) {
        const int pslot = w_it % kNumW;
        if (!wait_bar(p, sm.bar(B_WFULL + pslot), (w_it / kNumW) & 1, 0x4200)) return;
        if (pg == npages - 1) trace_stamp(p, gbase + i, 9);
        const uint32_t wpage = sm.w_page(pslot);
        const int kend = min(kc + cpp, nkc);
        for (uint32_t boff = 0; kc < kend; ++kc, boff += chunk_bytes) {
          const uint32_t ait = a_it + (uint32_t)kc;
          const int aslot = (int)(ait & (nA - 1));
          // later tiles of the task read the chunks the first tile waited for
          if (j == 0 && !wait_bar(p, sm.bar(B_AFULL + aslot), (ait >> lg) & 1, 0x4300)) return;
          if (kc == nkc - 1) trace_stamp(p, gbase + i, 10);
          tm_fence_after();
          const uint64_t ad = sdesc_sw128(sm.a_chunk(aslot, m128));
          const uint64_t bd = sdesc_sw128(wpage + boff);
#pragma unroll
          for (int k = 0; k < 4; ++k) tm_mma(d, ad + 2 * k, bd + 2 * k, idesc, (kc | k) != 0);
          if (last && kc + nA < nkc) tm_commit(sm.bar(B_AEMPTY + aslot));
        }
        if (j * npages + pg + kNumW < tot_pages) tm_commit(sm.bar(B_WEMPTY + pslot));
        w_it++;
      }
      tm_commit(sm.bar(B_ACCFULL + acc));
      trace_stamp(p, gbase + i, 12);
      acc_it++;
    }
    a_it += (uint32_t)nkc;
  }
}

__device__ void compute_role(const KParams& p, const FrameArgs& fa, const Task* tl, int n, int gbase, Sm sm,
                             uint32_t tmem, CState& st) {
  const int ct = threadIdx.x - kComputeBase;
  // Task records go through two shared-memory slots: while task i runs, the
  // leader copies record i+1 into the other slot (asynchronously, so its own
  // dependency wait is not held up); the barrier that ends every task orders
  // that copy before the next task's reads. A CTA on the critical path then
  // starts its next task without a round trip to L2.
  const uint32_t slot0 = sm.b + kSmemMisc + kMiscTask;
  const Task* slot = reinterpret_cast<const Task*>(sm.base + kSmemMisc + kMiscTask);
  if (ct == 0 && n > 0) {
    for (int q = 0; q < (int)sizeof(Task) / 16; ++q) cp_async16(slot0 + q * 16, reinterpret_cast<const uint8_t*>(tl) + q * 16);
    cp_async_wait_all();
  }
  csync();
  for (int i = 0; i < n; ++i) {
    const Task t = slot[i & 1];
    if (ct == 0 && i + 1 < n) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(tl + i + 1);
      const uint32_t dst = slot0 + (uint32_t)(((i + 1) & 1) * sizeof(Task));
      for (int q = 0; q < (int)sizeof(Task) / 16; ++q) cp_async16(dst + q * 16, src + q * 16);
    }
    const int gidx = gbase + i;
    st.gidx = gidx;
    if (ct == 0 && p.trace) p.trace[(size_t)gidx * kTraceStamps + 13] = INT64_MAX;
    bool ok = true;
    switch (t.type) {
      case T_PROJ: ok = proj_task(p, t, fa, sm, st, ct, gidx, tmem); break;
      case T_ATTN: ok = attn_task(p, t, fa, sm, st, ct, gidx); break;
      case T_DRAW: ok = draw_task(p, t, fa, sm, ct, gidx); break;
      case T_EMB0: ok = emb0_task(p, t, fa, ct, gidx); break;
      default: break;
    }
    if (!ok) break;
  }
  if (ct == 0) cp_async_wait_all();  // nothing may land after the CTA's teardown
}

__global__ void __launch_bounds__(kThreads, 1) frame_kernel(const __grid_constant__ KParams p) {
  extern __shared__ uint8_t smem_raw[];
  Sm sm;
  {
    const uint32_t a = saddr(smem_raw);
    const uint32_t pad = (1024 - (a & 1023)) & 1023;
    sm.base = smem_raw + pad;
    sm.b = a + pad;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* flag = reinterpret_cast<int32_t*>(sm.misc_u32(kMiscFlag));

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumW; ++i) { mb_init(sm.bar(B_WFULL + i), 1); mb_init(sm.bar(B_WEMPTY + i), 1); }
    // A full: the compute leader's (expect-tx) arrival; accumulator empty: one
    // per compute warp; receive full: the owner's expect-tx arrival plus the
    // bytes of the C partials; receive free: one arrival per owner in the cluster.
    for (int i = 0; i < kNumA; ++i) { mb_init(sm.bar(B_AFULL + i), 1); mb_init(sm.bar(B_AEMPTY + i), 1); }
    for (int i = 0; i < kNumAcc; ++i) {
      mb_init(sm.bar(B_ACCFULL + i), 1);
      mb_init(sm.bar(B_ACCEMPTY + i), 8);
    }
    for (int i = 0; i < 2; ++i) {
      mb_init(sm.bar(B_RFULL + i), 1 + kComputeThreads / 32);  // leader's byte count + each compute warp
      mb_init(sm.bar(B_RFREE + i), cluster_of(p));
    }
    mb_init(sm.bar(B_DRAIN), 1);
    mb_init(sm.bar(B_SCR), 1);
    mb_fence_init();
    flag[0] = *reinterpret_cast<volatile int32_t*>(p.status);  // a sticky error skips the frame
  }
  if (warp == 1) {
    tm_alloc(sm.b + kSmemMisc + kMiscTmem, kTmemCols);
    tm_relinquish();
  }
  tm_fence_before();
  __syncthreads();
  tm_fence_after();
  cluster_sync_all();
  const uint32_t tmem = *sm.misc_u32(kMiscTmem);
  const bool skip = flag[0] != 0;

  int lo, hi;
  if (p.mode == 0) {
    lo = p.phase_start[(size_t)blockIdx.x * (p.nph + 1) + p.phase_lo];
    hi = p.phase_start[(size_t)blockIdx.x * (p.nph + 1) + p.phase_hi];
  } else {
    lo = p.phase_start[(size_t)blockIdx.x * (p.nph + 1) + p.phase_lo];
    hi = p.phase_start[(size_t)blockIdx.x * (p.nph + 1) + p.phase_lo + 1];
  }
  const Task* tl = p.tasks + lo;
  const int n = skip ? 0 : hi - lo;

  uint32_t w_it = 0;
  CState st{};
  if (warp == 0) {
    if (lane == 0) producer_role(p, tl, n, lo, sm, w_it);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      mma_role(p, tl, n, lo, sm, tmem);
      tm_commit(sm.bar(B_DRAIN));  // every MMA issued by this thread is done when this arrives
      drain_bar(p, sm.bar(B_DRAIN), 0);
    }
    __syncwarp();
  } else if (warp >= kComputeBase / 32) {
    if (p.mode == 1) pdl_wait();
    FrameArgs fa = p.mode == 1 ? *p.fa_dev : p.fa;
    compute_role(p, fa, tl, n, lo, sm, tmem, st);
  }

  // Teardown after an abort: wait for this CTA's bulk copies still in flight.
  // Each slot's latest issue is the only one that can be pending, and its
  // barrier has not moved past that phase, so its parity names it.
  if (warp == 0 && lane == 0 && aborted(p)) {
    const uint32_t from = w_it > (uint32_t)kNumW ? w_it - kNumW : 0;
    for (uint32_t it = from; it < w_it; ++it) drain_bar(p, sm.bar(B_WFULL + it % kNumW), (it / kNumW) & 1);
  }
  if (threadIdx.x == kComputeBase && aborted(p)) {
    if (st.scr_it) drain_bar(p, sm.bar(B_SCR), (st.scr_it - 1) & 1);  // attention's copies
    const int lg = a_log2(p), nA = 1 << lg;
    for (uint32_t k = 1; k <= (uint32_t)nA && k <= st.a_it; ++k) {  // each slot's latest use
      const uint32_t it = st.a_it - k;
      if (st.a_bulk & (1u << (it & (nA - 1)))) drain_bar(p, sm.bar(B_AFULL + (it & (nA - 1))), (it >> lg) & 1);
    }
  }
  __syncthreads();
  if (p.mode == 1) pdl_trigger();
  cluster_sync_all();  // no peer writes into this CTA's shared memory after this
  if (warp == 1) {
    tm_fence_after();
    tm_dealloc(tmem, kTmemCols);
  }
  if (p.mode == 0 && p.last_launch) {
    if (threadIdx.x == 0) {
      __threadfence();
      const int old = atomicAdd(p.status + 2, 1);
      flag[1] = old == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (flag[1]) {  // the last CTA of the frame resets the counters for the next frame
      __threadfence();
      uint4* c4 = reinterpret_cast<uint4*>(p.counters);  // ncounters is a multiple of 4
      for (int i = threadIdx.x; i < p.ncounters / 4; i += blockDim.x) c4[i] = make_uint4(0u, 0u, 0u, 0u);
      if (threadIdx.x == 0) p.status[2] = 0;
      __threadfence();
    }
  }
}

#ifndef CP_SHAPE_1P7B

// ---------------------------------------------------------------- test kernels
__global__ void philox_test_kernel(const uint32_t* ctr, const uint32_t* key, int n, int use_curand,
                                   uint32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
  const uint2 k = make_uint2(key[2 * i], key[2 * i + 1]);
  const uint4 r = use_curand ? curand_Philox4x32_10(c, k) : philox10(c, k);
  out[4 * i] = r.x;
  out[4 * i + 1] = r.y;
  out[4 * i + 2] = r.z;
  out[4 * i + 3] = r.w;
}

__global__ void __launch_bounds__(kThreads, 1)
    draw_test_kernel(const float* logits, int V, const float* temp, const int32_t* topk, const float* topp,
                     const uint64_t* seed, const int64_t* offset, int group, int32_t* codes) {
  __shared__ __align__(16) uint8_t scratch[kDrawScratch];
  if (threadIdx.x < kComputeBase) return;  // the draw runs on the 256 compute threads, as in the frame
  const int ct = threadIdx.x - kComputeBase, row = blockIdx.x;
  draw_zero_hist(scratch, ct);
  gumbel_fill(reinterpret_cast<float*>(scratch + kDrawGumbel), V, seed[row], row, offset[row] + group, ct,
              kComputeThreads);
  csync();
  const int c = draw_row(logits + (size_t)row * V, V, temp[row], topk[row], topp[row], scratch, ct);
  if (ct == 0) codes[row] = c;
}

#endif  // !CP_SHAPE_1P7B

// ---------------------------------------------------------------- host side
const void* frame_kernel_fn() { return reinterpret_cast<const void*>(&frame_kernel); }

cudaError_t launch_frame(const KParams& prm, int grid, int cluster, int smem, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, frame_kernel, prm);
}

#ifndef CP_SHAPE_1P7B
cudaError_t launch_test_philox(const uint32_t* ctr, const uint32_t* key, int n, int use_curand, uint32_t* out,
                               cudaStream_t s) {
  philox_test_kernel<<<(n + 127) / 128, 128, 0, s>>>(ctr, key, n, use_curand, out);
  return cudaGetLastError();
}

cudaError_t launch_test_draw(const float* logits, int rows, int V, const float* temp, const int32_t* topk,
                             const float* topp, const uint64_t* seed, const int64_t* offset, int group,
                             int32_t* codes, cudaStream_t s) {
  draw_test_kernel<<<rows, kThreads, 0, s>>>(logits, V, temp, topk, topp, seed, offset, group, codes);
  return cudaGetLastError();
}
#endif  // !CP_SHAPE_1P7B

}  // namespace CP_BUILD
}  // namespace cp
