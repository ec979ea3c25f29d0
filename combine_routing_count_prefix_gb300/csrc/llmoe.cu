// llmoe.cu -- sm_103a kernels and the C ABI of libllmoe.so (see include/llmoe.h).
//
// One GPU holds R simulated expert-parallel ranks as R segments of one
// allocation, each laid out as LLMoEBufferLayout<T> (LL_MoE_Buffers.hpp) for
// a payload type T of bf16, fp16 or fp32.  The data path is data movement plus
// one fp32 multiply-add per value in the combine, so it is bound by HBM
// bandwidth and latency: 16-byte accesses, no tensor cores (nothing here is a
// dense contraction).  Every launch uses programmatic dependent launch.
//
// Kernels:
//   route scan (route_hist / route_slot, the prologue of the route, dispatch,
//     combine, put and signalled kernels): per-(expert, source rank) counts
//     and slots, where the slot of token t for expert e is the number of
//     earlier tokens of the same source rank that chose e.  A shared-memory
//     histogram of the tokens before the CTA's block (integer atomics: the
//     result does not depend on their order) plus an in-block rank; no
//     global atomics and no scratch memory.
//   dispatch_kernel<kRows>: one producer lane streams the CTA's x rows into a
//     shared-memory ring (cp.async.bulk, mbarrier); each consumer thread owns a
//     16-byte quad of a chunk and writes it to the token's K messages.  A
//     message is 4 + H * sizeof(T) bytes, 4 (mod 16) when H * sizeof(T) is a
//     multiple of 16, so a destination starts at any 4-byte phase: the quad is
//     shifted by whole 32-bit words and stored aligned, with 4/8-byte stores
//     only at a message's head and tail.  With kRows the quad also goes, as it
//     is, to the entry's row of the experts' input (llmoe_dispatch_unpack).
//   combine_kernel<T>: each warp reduces 32 quads of one output row: up to 8
//     aligned 16-byte loads of expert rows, fp32 products rounded then added
//     in ascending k (__fmul_rn / __fadd_rn: never contracted to an FMA), the
//     sum stored as T (bf16 / fp16 rounded to nearest even).
//   combine_put_kernel, combine_reduce_ring_kernel<T> / combine_reduce_kernel<T>:
//     the staged combine through the combine receive buffers (messages written
//     with realigned stores; read back through a shared-memory ring of bulk
//     copies for large grids, or at their own 4-byte alignment into registers
//     for small ones).
//   unpack_balanced_kernel, unpack_kernel: received messages to the experts'
//     input layout, driven by the count words.
//   dispatch_signaled_kernel: dispatch and unpack in one cooperative launch;
//     producers raise each source's count words, consumer CTAs grouped by
//     source wait for them (bounded) and unpack an equal share of its rows.
//   clean_kernel: zeroes a set's R * E signal words (LLMoEBuffer::clean_meta).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <climits>

#include "llmoe.h"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxTokensPerBlock = 32;

struct Geometry {
  uint8_t* base;         // rank 0's buffer
  uint64_t rank_stride;  // bytes between rank buffers
  uint64_t recv_off;     // this set's receive region, from a rank buffer's start
  uint64_t sig_off;      // this set's signal words
  uint64_t other_sig_off;  // the other set's signal words
  uint64_t msg;          // 4 + H * sizeof(T)
  int32_t* err;          // optional error word
  uint32_t flags;        // LLMOE_FLAG_*
  int T_max, T, H, R, E, K, L;
  uint32_t L_mul;  // ceil(2^32 / L) (0 for L = 1): e / L = umulhi(e, L_mul) for every expert id e < 2^16
  int dtype;      // LLMOE_DTYPE_*
  int row_bytes;  // H * element size
  int nq;       // 16-byte quads per row
  int nchunks;  // warp units per row, ceil(nq / 32)
  int TB;       // tokens per CTA
  int nblk;     // token blocks per source rank
  int dsplit;   // dispatch: data CTAs per token block (each a share of the rows' ring chunks)
  int csplit;   // combine: data CTAs per token block (each a share of the rows' 512 B chunks)
  int pf_units; // combine: units per warp whose expert rows are prefetched into L2 before the wait
};

__device__ __forceinline__ void report(int32_t* err, int32_t code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// Phase trace, compiled in only with -DLLMOE_PHASE_TRACE=1 (a separate build
// of the library; the normal build has none of it).  A traced kernel stamps
// the global nanosecond timer and its SM's cycle counter at fixed points of
// its prologue and data phase into a per-CTA row of a device array (the
// dispatch's CTAs from row 0, the combine's from row kTraceCtas / 2, so one
// round of both is traced at once), which llmoe_phase_trace_read copies
// out.  Used to find where a kernel's fixed latency goes.
#ifndef LLMOE_PHASE_TRACE
#define LLMOE_PHASE_TRACE 0
#endif
#if LLMOE_PHASE_TRACE
constexpr int kTraceCtas = 65536;  // rows: dispatch CTAs from 0, combine CTAs from kTraceCtas / 2
constexpr int kTracePhases = 8;   // per CTA: kTracePhases timer stamps, kTracePhases cycle stamps
__device__ unsigned long long g_phase_trace[kTraceCtas * 2 * kTracePhases];
// The cycle slot of phase 0 holds the CTA's SM id instead.
__device__ __forceinline__ void trace_phase(int base, int p) {
  const int row = base + (int)blockIdx.x;
  if (row < kTraceCtas) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    g_phase_trace[(size_t)row * 2 * kTracePhases + p] = t;
    unsigned long long c = (unsigned long long)clock64();
    if (p == 0) {
      unsigned smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      c = smid;
    }
    g_phase_trace[(size_t)row * 2 * kTracePhases + kTracePhases + p] = c;
  }
}
#define TRACE(p, cond)             \
  do {                             \
    if (cond) trace_phase(0, p);   \
  } while (0)
#define TRACE_C(p, cond)                          \
  do {                                            \
    if (cond) trace_phase(kTraceCtas / 2, p);     \
  } while (0)
#else
#define TRACE(p, cond) \
  do {                 \
  } while (0)
#define TRACE_C(p, cond) \
  do {                   \
  } while (0)
#endif

// Programmatic dependent launch: every kernel here is launched so that it may
// start while the previous kernel on the stream drains.  Each kernel first
// lets the next kernel on the stream begin launching (that kernel still waits
// for this one before it touches memory), then waits for the previous grid to
// complete and flush before its first global memory access (a no-op when
// launched without the attribute).  With LLMOE_FLAG_INPUTS_READY, dispatch
// and combine read their routing inputs before that wait.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void release_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Shared-memory view of the route scan.
struct RouteSmem {
  int* hist;  // [E] tokens before the block (then: all tokens) per expert
  int* ent;   // [TB*K] the block's expert ids (-1 masked or invalid)
  int* slot;  // [TB*K] slot per block entry, -1 if none
};

__device__ __forceinline__ RouteSmem carve_route(unsigned char* smem, const Geometry& g) {
  RouteSmem s;
  s.hist = reinterpret_cast<int*>(smem);
  s.ent = s.hist + g.E;
  s.slot = s.ent + g.TB * g.K;
  return s;
}

// Routing count / prefix scan for tokens [t0, t1) of source rank src, in two
// steps.  route_hist loads the block's entries into s.ent and builds s.hist =
// per-expert entries of the tokens before the block (returns after a
// barrier).  route_slot(q) then gives entry q's slot: hist[e] plus the
// earlier in-block tokens choosing e; each thread calls it for its own
// entries, so a kernel can turn slots into addresses in the same pass.
// route_count_block adds the block's entries to s.hist (full counts, for the
// CTA of a source rank's last block); its caller syncs before reading them.
// route_hist runs on threads [0, nthr) of the CTA numbered by tid, which meet
// at Sync() (a __syncthreads, or a named barrier of a subset of warps).
//
// Every CTA of a launch runs this prologue at the same moment, so its cost is
// the instructions all their warps issue as much as its latency: one
// shared-memory atomic per id, kPrefetch ids in flight per thread (one memory
// round trip for up to kPrefetch * nthr ids), and the per-entry slot work on
// one thread per entry.
constexpr int kPrefetch = 8;  // prefix ids a thread has in flight per pass

__device__ __forceinline__ void sync_all() { __syncthreads(); }

template <void (*Sync)() = sync_all>
__device__ void route_hist(const Geometry& g, const int64_t* __restrict__ idx, int src, int t0, int t1,
                           const RouteSmem& s, int tid, int nthr) {
  const int K = g.K, E = g.E;
  const int64_t* src_idx = idx + (int64_t)src * g.T * K;
  const int npre = t0 * K, nblock = (t1 - t0) * K;
  // the first pass of prefix loads is issued before anything else
  int64_t pre[kPrefetch];
#pragma unroll
  for (int j = 0; j < kPrefetch; ++j) {
    const int i = tid + j * nthr;
    pre[j] = i < npre ? src_idx[i] : -1;
  }
  for (int e = tid; e < E; e += nthr) s.hist[e] = 0;
  for (int q = tid; q < nblock; q += nthr) {
    const int64_t e = src_idx[npre + q];
    s.ent[q] = (e >= 0 && e < E) ? (int)e : -1;
    if (e < -1 || e >= E) report(g.err, LLMOE_DEV_BAD_EXPERT);
  }
  Sync();
  for (int base = 0;;) {
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j)
      if (pre[j] >= 0 && pre[j] < E) atomicAdd(&s.hist[pre[j]], 1);
    base += kPrefetch * nthr;
    if (base >= npre) break;
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j) {
      const int i = base + tid + j * nthr;
      pre[j] = i < npre ? src_idx[i] : -1;
    }
  }
  Sync();
}

__device__ __forceinline__ int route_slot(const Geometry& g, const RouteSmem& s, int q) {
  const int e = s.ent[q];
  if (e < 0) return -1;
  int r = 0, tl = 0, k = q;  // one token per CTA: entry q is the token's k-th
  if (g.TB > 1) {
    tl = q / g.K;
    k = q - tl * g.K;
    for (int p = 0; p < tl * g.K; ++p) r += (s.ent[p] == e);  // earlier tokens of the block
  }
  if (g.err != nullptr)  // validate mode: an expert twice in one token
    for (int k2 = 0; k2 < k; ++k2)
      if (s.ent[tl * g.K + k2] == e) report(g.err, LLMOE_DEV_DUPLICATE);
  const int sl = s.hist[e] + r;
  if (sl >= g.T_max) {  // only reachable when a token repeats an expert
    report(g.err, LLMOE_DEV_SLOT_RANGE);
    return -1;
  }
  return sl;
}

// After every thread's route_slot calls (i.e. after a __syncthreads).
__device__ __forceinline__ void route_count_block(const RouteSmem& s, int nblock) {
  for (int q = threadIdx.x; q < nblock; q += blockDim.x)
    if (s.ent[q] >= 0) atomicAdd(&s.hist[s.ent[q]], 1);
}

// Owner of expert e: rank e / L, local expert e % L, without a division.
__device__ __forceinline__ int owner_rank(const Geometry& g, int e) {
  return g.L_mul == 0 ? e : (int)__umulhi((unsigned)e, g.L_mul);
}

// Zeroes the other buffer set's R * E signal words (LLMOE_FLAG_CLEAN_OTHER_SET:
// the clean that the next call on that set needs), words first, first +
// stride, ...; called after the kernel has waited for the previous one.
__device__ __forceinline__ void clean_other_set(const Geometry& g, int64_t first, int64_t stride) {
  if ((g.flags & LLMOE_FLAG_CLEAN_OTHER_SET) == 0) return;
  const int64_t n = (int64_t)g.R * g.E;
  for (int64_t i = first; i < n; i += stride) {
    const int64_t r = i / g.E, e = i % g.E;
    reinterpret_cast<int64_t*>(g.base + r * g.rank_stride + g.other_sig_off)[e] = 0;
  }
}
__device__ __forceinline__ void clean_other_set(const Geometry& g) {
  clean_other_set(g, blockIdx.x * (int64_t)blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
}

// Writes rank dst's (dispatch) or rank src's (combine) signal words from the
// full histogram; checks that each word was zero (cleaned) in validate mode.
__device__ __forceinline__ void put_signal(const Geometry& g, int64_t* word, int value) {
  if (g.err != nullptr && *reinterpret_cast<volatile int64_t*>(word) != 0) report(g.err, LLMOE_DEV_STALE_SIGNAL);
  *word = (int64_t)value;
}

// The first R CTAs of a dispatch or combine grid are count CTAs, one per
// source rank src: the per-expert counts of all of src's tokens (the
// histogram of its ids) become the signal words (dispatch: rank e / L's word
// (e % L) * R + src = the count of bucket (e, src); combine: rank src's word e
// = rows expert e returns to src), and the count CTAs together zero the other
// set's words when LLMOE_FLAG_CLEAN_OTHER_SET asks for it.  They move no rows,
// so no data CTA carries the counts after its rows.
__device__ void count_source(const Geometry& g, const int64_t* __restrict__ idx, int src, const RouteSmem& s,
                             bool early, bool dispatch_words) {
  release_next_grid();
  if (!early) wait_prior_grid();
  route_hist(g, idx, src, g.T, g.T, s, threadIdx.x, blockDim.x);  // all tokens: the full counts
  if (early) wait_prior_grid();  // the signal words may be in use until now
  clean_other_set(g, (int64_t)src * blockDim.x + threadIdx.x, (int64_t)g.R * blockDim.x);
  for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
    int64_t* w = dispatch_words
                     ? reinterpret_cast<int64_t*>(g.base + (e / g.L) * g.rank_stride + g.sig_off) +
                           ((int64_t)(e % g.L) * g.R + src)
                     : reinterpret_cast<int64_t*>(g.base + src * g.rank_stride + g.sig_off) + e;
    put_signal(g, w, s.hist[e]);
  }
}

// Destination quad from the previous and current source quads when the
// payload starts `phase` words past a 16-byte boundary.
__device__ __forceinline__ uint4 shift_words(const uint4& prev, const uint4& cur, int phase) {
  switch (phase) {
    case 0: return cur;
    case 1: return make_uint4(prev.w, cur.x, cur.y, cur.z);
    case 2: return make_uint4(prev.z, prev.w, cur.x, cur.y);
    default: return make_uint4(prev.y, prev.z, prev.w, cur.x);
  }
}

// 16-byte read-only load that does not allocate in L1: for rows read exactly
// once (expert outputs in the combine and the staged put), where L1 lines
// would only add allocation work to every miss.
__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ void st16(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void st8(uint8_t* p, uint32_t a, uint32_t b) {
  *reinterpret_cast<uint2*>(p) = make_uint2(a, b);
}
__device__ __forceinline__ void st4(uint8_t* p, uint32_t a) { *reinterpret_cast<uint32_t*>(p) = a; }

// Writes source quad j of a token row (and the header / tail pieces that fall
// to it) into the message at `dest` (pack_dest).  prev is quad j-1, or
// (0,0,0,t) for j == 0 so that prev.w is the header.
// A message destination packed into one word: the 16-byte-aligned address
// qb at or below the payload start, OR the payload's 4-byte phase (0..3).
__device__ __forceinline__ uintptr_t pack_dest(uint8_t* msg_addr) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(msg_addr) + 4;
  return (pa & ~(uintptr_t)15) | ((pa >> 2) & 3);
}

__device__ __forceinline__ void put_quad(uintptr_t dest, int j, int nq, const uint4& prev, const uint4& cur) {
  const int phase = (int)(dest & 3);
  uint8_t* qb = reinterpret_cast<uint8_t*>(dest & ~(uintptr_t)15);  // 16-byte aligned
  uint8_t* pa = qb + 4 * phase;                                       // payload
  if (j > 0) {
    st16(qb + 16 * j, shift_words(prev, cur, phase));
  } else {
    switch (phase) {
      case 0: st16(qb, cur); st4(pa - 4, prev.w); break;
      case 1: st16(qb, shift_words(prev, cur, 1)); break;
      case 2: st4(qb + 4, prev.w); st8(qb + 8, cur.x, cur.y); break;
      default: st8(qb + 8, prev.w, cur.x); break;
    }
  }
  if (j == nq - 1 && phase != 0) {
    uint8_t* tq = qb + 16 * (size_t)nq;
    switch (phase) {
      case 1: st4(tq, cur.w); break;
      case 2: st8(tq, cur.z, cur.w); break;
      default: st8(tq, cur.y, cur.z); st4(tq + 8, cur.w); break;
    }
  }
}

// ---------------------------------------------------------------------------
// Asynchronous bulk copies into a shared-memory ring (cp.async.bulk with
// mbarrier completion).  One producer lane keeps up to kStages chunks in
// flight per CTA without holding them in registers; consumer warps wait on a
// stage's "full" barrier, use it, and arrive on its "empty" barrier so the
// producer can refill it.  Every wait is bounded (kSpinLimit clock cycles,
// about one second): on expiry the kernel records LLMOE_DEV_TIMEOUT, stops
// issuing, and drains the copies it has in flight before it returns.
// ---------------------------------------------------------------------------
constexpr long long kSpinLimit = 2000000000LL;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Waits for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > kSpinLimit) {
      report(err, LLMOE_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}
// global -> shared bulk copy; both addresses 16-byte aligned, bytes % 16 == 0
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// The ring: kStages stages of stage_bytes each, plus full / empty barriers.
template <int kStages>
struct Ring {
  uint8_t* data;
  uint64_t* full;
  uint64_t* empty;
  uint32_t stage_bytes;
  __device__ uint8_t* stage(int s) const { return data + (size_t)s * stage_bytes; }
};

// Producer-side bookkeeping shared with the drain at the end of a kernel.
struct RingState {
  int issued;    // stages handed to the copy engine
  int consumed;  // lowest stage count every consumer warp got through
};

// After a timeout: wait (bounded) for every issued stage nobody consumed, so
// no copy is still writing this CTA's shared memory when it exits.
template <int kStages>
__device__ void ring_drain(const Ring<kStages>& r, const RingState& st, int32_t* err) {
  for (int it = st.consumed; it < st.issued; ++it) {
    const int s = it % kStages;
    if (!mbar_wait(&r.full[s], (it / kStages) & 1, err)) return;
  }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
// Ring shapes (compile-time tuning parameters).
#ifndef LLMOE_DSP_CONSUMERS
#define LLMOE_DSP_CONSUMERS 4
#endif
#ifndef LLMOE_DSP_STAGES
#define LLMOE_DSP_STAGES 8
#endif
#ifndef LLMOE_CMB_THREADS
#define LLMOE_CMB_THREADS 128
#endif
#ifndef LLMOE_CMB_PREFETCH_BYTES
#define LLMOE_CMB_PREFETCH_BYTES (16 << 20)  // expert-row bytes a combine prefetches into L2 before its wait
#endif

constexpr int kDspConsumers = LLMOE_DSP_CONSUMERS;   // warps; lanes x 16 B = one chunk
constexpr int kDspChunk = kDspConsumers * 32 * 16;   // x bytes per stage
constexpr int kDspStageBytes = kDspChunk + 16;       // + the quad before the chunk
constexpr int kDspStages = LLMOE_DSP_STAGES;
constexpr int kDspThreads = 32 * (1 + kDspConsumers);
// A grid with several tokens per CTA (TB > 1: more tokens than one wave of
// CTAs, e.g. 8 ranks x 1,024 tokens) is split further: each token block gets
// up to LLMOE_DSP_SPLIT dispatch CTAs (one per 2 KB ring chunk of its rows) and,
// from 4 tokens per block, LLMOE_CMB_SPLIT combine CTAs, each moving a
// contiguous share of the rows' chunks.  The grid then spans many waves and the CTA scheduler gives the SMs
// that move rows fastest more CTAs: a GB300's SMs do not move rows at one rate
// (per-SM rates measured in the dispatch differ by up to 1.9x, in groups of
// SMs), and with one wave of equal CTAs the slowest group sets the kernel's
// end.  With one token per CTA the split only repeats the route scan.
#ifndef LLMOE_DSP_SPLIT
#define LLMOE_DSP_SPLIT 64
#endif
#ifndef LLMOE_CMB_SPLIT
#define LLMOE_CMB_SPLIT 2
#endif

// Named barrier of the consumer warps of a dispatch CTA (the producer warp
// streams x and does not take part in the route scan).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDspConsumers * 32) : "memory");
}

// Grid: R count CTAs (count_source), then R * nblk data CTAs, data CTA
// (src, b) owning tokens [b * TB, b * TB + TB) of source rank src.  Warp 0
// is the producer: its lane 0 streams the CTA's x rows into the ring from
// the start.  The consumer warps meanwhile run the route scan among
// themselves (named barrier) and pack the destinations into shared memory,
// then take the ring's chunks.
// kRows: the CTA also writes each entry's row of the experts' input, recv_x
// row (e * R + src) * T_max + slot and recv_src there = t, which is what
// llmoe_unpack makes from the messages: the CTA holds the row and knows the
// slot, so it stores the row as it is (aligned) beside the message.
template <bool kRows>
__global__ void __launch_bounds__(kDspThreads, 8) dispatch_kernel(Geometry g, const void* __restrict__ x,
                                                               const int64_t* __restrict__ idx,
                                                               void* __restrict__ recv_x,
                                                               int32_t* __restrict__ recv_src) {
  extern __shared__ __align__(128) unsigned char smem[];
  Ring<kDspStages> ring;
  ring.data = smem;
  ring.stage_bytes = kDspStageBytes;
  ring.full = reinterpret_cast<uint64_t*>(smem + kDspStages * kDspStageBytes);
  ring.empty = ring.full + kDspStages;
  __shared__ RingState st;
  const RouteSmem s = carve_route(reinterpret_cast<unsigned char*>(ring.empty + kDspStages), g);
  uintptr_t* s_dst = reinterpret_cast<uintptr_t*>(s.slot + g.TB * g.K + (g.E & 1));
  uint4** s_xrow = reinterpret_cast<uint4**>(s_dst + g.TB * g.K);  // kRows: the entries' recv_x rows
  const bool early = (g.flags & LLMOE_FLAG_INPUTS_READY) != 0;
  if ((int)blockIdx.x < g.R) {
    count_source(g, idx, blockIdx.x, s, early, true);
    return;
  }

  const int bid = (int)blockIdx.x - g.R;
  const int part = bid % g.dsplit;
  const int src = bid / g.dsplit / g.nblk, b = bid / g.dsplit % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_bytes = g.row_bytes;
  const int nch_row = (row_bytes + kDspChunk - 1) / kDspChunk;
  const int c0 = nch_row * part / g.dsplit;  // this CTA's chunks [c0, c0 + nch) of each of its rows
  const int nch = nch_row * (part + 1) / g.dsplit - c0;
  const int n_iters = (t1 - t0) * nch;
  TRACE(0, threadIdx.x == 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDspStages; ++i) {
      mbar_init(&ring.full[i], 1);
      mbar_init(&ring.empty[i], kDspConsumers);
    }
    mbar_init_fence();
    st.issued = 0;
    st.consumed = INT_MAX;
  }
  release_next_grid();
  if (!early) wait_prior_grid();
  TRACE(1, threadIdx.x == 0);
  __syncthreads();  // barriers initialised

  if (warp == 0) {
    // producer: x does not depend on the routing, so it streams from the start
    if (lane == 0) {
      const uint8_t* xsrc = reinterpret_cast<const uint8_t*>(x) + ((int64_t)src * g.T + t0) * row_bytes;
      int next = 0;
      for (; next < n_iters; ++next) {
        const int sidx = next % kDspStages, use = next / kDspStages;
        if (use > 0 && !mbar_wait(&ring.empty[sidx], (use - 1) & 1, g.err)) break;
        const int tl = next / nch, c = c0 + next % nch;
        const int len = min(kDspChunk, row_bytes - c * kDspChunk);
        uint8_t* dst = ring.stage(sidx);
        const uint8_t* row = xsrc + (size_t)tl * row_bytes;
        if (c == 0) {
          mbar_arrive_expect_tx(&ring.full[sidx], len);
          bulk_load(dst + 16, row, len, &ring.full[sidx]);
        } else {
          mbar_arrive_expect_tx(&ring.full[sidx], len + 16);
          bulk_load(dst, row + c * kDspChunk - 16, len + 16, &ring.full[sidx]);
        }
      }
      st.issued = next;
    }
    __syncwarp();  // the warp meets the CTA barrier below converged
  } else {
    const int ct = threadIdx.x - 32;  // the 16-byte quad of the chunk this thread moves
    route_hist<consumers_sync>(g, idx, src, t0, t1, s, ct, kDspConsumers * 32);
    TRACE(2, threadIdx.x == 32);
    const int nblock = (t1 - t0) * g.K;
    for (int q = ct; q < nblock; q += kDspConsumers * 32) {
      const int e = s.ent[q], sl = route_slot(g, s, q);
      uintptr_t d = 0;
      uint4* xr = nullptr;
      if (sl >= 0) {
        const int dst = owner_rank(g, e), le = e - dst * g.L;
        const uint64_t row = ((uint64_t)le * g.R + src) * g.T_max + sl;
        d = pack_dest(g.base + dst * g.rank_stride + g.recv_off + row * g.msg);
        if constexpr (kRows) {
          const int64_t orow = ((int64_t)e * g.R + src) * g.T_max + sl;
          xr = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(recv_x) + orow * row_bytes);
          if (part == 0) recv_src[orow] = t0 + q / g.K;
        }
      }
      s_dst[q] = d;
      if constexpr (kRows) s_xrow[q] = xr;
    }
    consumers_sync();
    TRACE(3, threadIdx.x == 32);
    if (early) wait_prior_grid();  // the receive rows may be in use until now
    TRACE(4, threadIdx.x == 32);
    int it = 0;
    for (; it < n_iters; ++it) {
      const int sidx = it % kDspStages;
      if (!mbar_wait(&ring.full[sidx], (it / kDspStages) & 1, g.err)) break;
      TRACE(5, threadIdx.x == 32 && it == 0);
      const int tl = it / nch, c = c0 + it % nch;
      const int len = min(kDspChunk, row_bytes - c * kDspChunk);
      const uint8_t* sb = ring.stage(sidx);
      // the token's destinations from shared memory, one put_quad in a loop:
      // unrolling the destinations into registers made the loop's code so
      // much larger that its first pass, from cold instruction caches, cost
      // more than the loads it saved (tiny workload 0.9 us a round)
      const uintptr_t* dsts = s_dst + tl * g.K;
      if (ct * 16 < len) {
        const uint4 cur = *reinterpret_cast<const uint4*>(sb + 16 + 16 * ct);
        const uint4 prev = (c == 0 && ct == 0) ? make_uint4(0, 0, 0, (uint32_t)(t0 + tl))
                                               : *reinterpret_cast<const uint4*>(sb + 16 * ct);
        const int j = c * (kDspChunk / 16) + ct;
        for (int k = 0; k < g.K; ++k) {
          const uintptr_t d = dsts[k];
          if (d != 0) put_quad(d, j, g.nq, prev, cur);
          if constexpr (kRows) {
            uint4* xr = s_xrow[tl * g.K + k];
            if (xr != nullptr) xr[j] = cur;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ring.empty[sidx]);
    }
    if (lane == 0) atomicMin(&st.consumed, it);
    TRACE(6, threadIdx.x == 32);
  }
  __syncthreads();
  if (st.consumed < st.issued) ring_drain(ring, st, g.err);
  TRACE(7, threadIdx.x == 0);
}

// ---------------------------------------------------------------------------
// combine
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

#ifndef LLMOE_PACKED_F32X2
#define LLMOE_PACKED_F32X2 1
#endif
#if LLMOE_PACKED_F32X2
// Both products in one instruction (mul.rn.f32x2: each lane rounded as
// __fmul_rn rounds it), then the two sums as separate __fadd_rn.  A packed
// add after the packed multiply is fused into one packed FMA by the
// assembler, which changes the rounding, so the sums stay scalar.
__device__ __forceinline__ void axpy2(float& a0, float& a1, float w, float y0, float y1) {
  float p0, p1;
  asm("{\n\t.reg .b64 y, w2;\n\tmov.b64 y, {%2, %3};\n\tmov.b64 w2, {%4, %4};\n\t"
      "mul.rn.f32x2 y, y, w2;\n\tmov.b64 {%0, %1}, y;\n\t}"
      : "=f"(p0), "=f"(p1)
      : "f"(y0), "f"(y1), "f"(w));
  a0 = __fadd_rn(a0, p0);
  a1 = __fadd_rn(a1, p1);
}
#else
__device__ __forceinline__ void axpy2(float& a0, float& a1, float w, float y0, float y1) {
  a0 = __fadd_rn(a0, __fmul_rn(w, y0));
  a1 = __fadd_rn(a1, __fmul_rn(w, y1));
}
#endif

// One 16-byte quad of payload values, by payload type: accumulate w * value
// into acc in fp32 (product rounded, then sum rounded: never fused), and pack
// the accumulators back (bf16 / fp16 round to nearest even; fp32 kept).
template <int DT>
__device__ __forceinline__ void axpy_q(float (&acc)[8], float w, const uint4& v);
template <>
__device__ __forceinline__ void axpy_q<LLMOE_DTYPE_BF16>(float (&acc)[8], float w, const uint4& v) {
  axpy2(acc[0], acc[1], w, bf16lo(v.x), bf16hi(v.x));
  axpy2(acc[2], acc[3], w, bf16lo(v.y), bf16hi(v.y));
  axpy2(acc[4], acc[5], w, bf16lo(v.z), bf16hi(v.z));
  axpy2(acc[6], acc[7], w, bf16lo(v.w), bf16hi(v.w));
}
template <>
__device__ __forceinline__ void axpy_q<LLMOE_DTYPE_FP16>(float (&acc)[8], float w, const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));  // exact
    axpy2(acc[2 * i], acc[2 * i + 1], w, f.x, f.y);
  }
}
template <>
__device__ __forceinline__ void axpy_q<LLMOE_DTYPE_FP32>(float (&acc)[8], float w, const uint4& v) {
  axpy2(acc[0], acc[1], w, __uint_as_float(v.x), __uint_as_float(v.y));
  axpy2(acc[2], acc[3], w, __uint_as_float(v.z), __uint_as_float(v.w));
}

template <int DT>
__device__ __forceinline__ uint4 pack_q(const float (&acc)[8]) {
  if constexpr (DT == LLMOE_DTYPE_FP32) {
    return make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                      __float_as_uint(acc[3]));
  } else {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (DT == LLMOE_DTYPE_FP16) {
        const __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
        u[i] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        u[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
      }
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
}

constexpr int kCmbThreads = LLMOE_CMB_THREADS;
constexpr int kCmbWarps = kCmbThreads / 32;
constexpr int kKBatch = 8;  // most expert-row loads a lane has in flight

// Grid: R count CTAs (count_source: the flag words), then R * nblk data CTAs.
// A data CTA reduces tokens [t0, t1) of source rank src; one warp reduces 32
// quads (512 B) of one output row per unit: up to kKBatch expert rows are
// loaded (16 B per lane each) before they are accumulated, in ascending k.
template <int DT, int KB>  // KB: expert-row loads in flight per lane, the top-k rounded up to 2, 4 or 8
__global__ void __launch_bounds__(kCmbThreads) combine_kernel(Geometry g, const void* __restrict__ y,
                                                              const int64_t* __restrict__ idx,
                                                              const float* __restrict__ topk_w,
                                                              void* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  const int TBK = g.TB * g.K;
  const uint4** s_row = reinterpret_cast<const uint4**>(s.slot + TBK + (g.E & 1));
  float* s_w = reinterpret_cast<float*>(s_row + TBK);
  const bool early = (g.flags & LLMOE_FLAG_INPUTS_READY) != 0;
  if ((int)blockIdx.x < g.R) {
    count_source(g, idx, blockIdx.x, s, early, false);
    return;
  }

  const int bid = (int)blockIdx.x - g.R;
  const int part = bid % g.csplit;
  const int src = bid / g.csplit / g.nblk, b = bid / g.csplit % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const int nblock = (t1 - t0) * g.K;
  const float* wblk = topk_w + ((int64_t)src * g.T + t0) * g.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TRACE_C(0, threadIdx.x == 0);
  release_next_grid();
  if (!early) wait_prior_grid();
  TRACE_C(1, threadIdx.x == 0);
  const float w0 = threadIdx.x < nblock ? wblk[threadIdx.x] : 0.0f;  // before the prologue's barriers
  route_hist(g, idx, src, t0, t1, s, threadIdx.x, blockDim.x);
  TRACE_C(2, threadIdx.x == 0);
  for (int q = threadIdx.x; q < nblock; q += blockDim.x) {
    const int e = s.ent[q], sl = route_slot(g, s, q);
    const uint4* r = nullptr;
    if (sl >= 0) {
      const uint64_t row = (uint64_t)e * g.R * g.T_max + (uint64_t)src * g.T_max + sl;
      r = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(y) + row * g.row_bytes);
    }
    s_row[q] = r;
    s_w[q] = q == threadIdx.x ? w0 : wblk[q];
  }
  __syncthreads();
  TRACE_C(3, threadIdx.x == 0);
  if (early) {
    // While the previous kernel drains, pull the expert rows of each warp's
    // first units into L2.  A prefetch reads nothing into the kernel: if the
    // previous kernel is still writing y, its stores update the same L2 lines
    // (L2 is where the device's memory is kept coherent), and the loads below
    // come after the wait.
    const int nunits = (t1 - t0) * g.nchunks;
    for (int u = warp; u < nunits && u < warp + g.pf_units * kCmbWarps; u += kCmbWarps) {
      // lane k: one bulk prefetch of the unit's 512 B of row k (one instruction
      // per row, where a prefetch per lane and 16 bytes took 32; DS-V3 round
      // 49.2 -> 49.0 us, many-small 13.1 -> 13.0; without any 50.5 and 13.9)
      const int tl = u / g.nchunks, c = u % g.nchunks;
      const uint32_t bytes = (uint32_t)min(512, g.row_bytes - 512 * c);
      if (lane < g.K) {
        const uint4* r = s_row[tl * g.K + lane];
        if (r != nullptr)
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(r + c * 32), "r"(bytes) : "memory");
      }
    }
    wait_prior_grid();  // y may come from the previous kernel
  }
  TRACE_C(4, threadIdx.x == 0);

  const int c0 = g.nchunks * part / g.csplit, cn = g.nchunks * (part + 1) / g.csplit - c0;  // this CTA's chunks
  const int nunits = (t1 - t0) * cn;
  for (int u = warp; u < nunits; u += kCmbWarps) {
    const int tl = u / cn, c = c0 + u % cn;
    const int t = t0 + tl;
    const int j = c * 32 + lane;
    if (j >= g.nq) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const uint4* const* trows = s_row + tl * g.K;
    const float* tws = s_w + tl * g.K;
    for (int k0 = 0; k0 < g.K; k0 += KB) {
      uint4 v[KB];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int k = k0 + i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (k < g.K && trows[k] != nullptr) v[i] = ld_stream16(trows[k] + j);
      }
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int k = k0 + i;
        if (k < g.K && trows[k] != nullptr) axpy_q<DT>(acc, tws[k], v[i]);
      }
    }
    reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) + ((int64_t)src * g.T + t) * g.row_bytes)[j] =
        pack_q<DT>(acc);
    TRACE_C(5, threadIdx.x == 0 && u == warp);
  }
  TRACE_C(6, threadIdx.x == 0);
  TRACE_C(7, threadIdx.x == 0);
}

// ---------------------------------------------------------------------------
// staged combine: put the expert output rows as messages into the source
// ranks' combine receive regions, then reduce from them
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 shfl_up16(const uint4& v) {
  return make_uint4(__shfl_up_sync(0xffffffffu, v.x, 1), __shfl_up_sync(0xffffffffu, v.y, 1),
                    __shfl_up_sync(0xffffffffu, v.z, 1), __shfl_up_sync(0xffffffffu, v.w, 1));
}
__device__ __forceinline__ uint4 shfl_down16(const uint4& v) {
  return make_uint4(__shfl_down_sync(0xffffffffu, v.x, 1), __shfl_down_sync(0xffffffffu, v.y, 1),
                    __shfl_down_sync(0xffffffffu, v.z, 1), __shfl_down_sync(0xffffffffu, v.w, 1));
}
__device__ __forceinline__ uint4 shfl_idx16(const uint4& v, int src_lane) {
  return make_uint4(__shfl_sync(0xffffffffu, v.x, src_lane), __shfl_sync(0xffffffffu, v.y, src_lane),
                    __shfl_sync(0xffffffffu, v.z, src_lane), __shfl_sync(0xffffffffu, v.w, src_lane));
}

// Rows move in steps of up to kRowBatch 512-byte chunks per warp (unpack) or kPutBatch (staged put).
#ifndef LLMOE_ROW_BATCH
#define LLMOE_ROW_BATCH 8
#endif
#ifndef LLMOE_UNPACK_MIN_BLOCKS
#define LLMOE_UNPACK_MIN_BLOCKS 4
#endif
constexpr int kRowBatch = LLMOE_ROW_BATCH;
// The staged put's token blocks are sized for two waves of CTAs, not one:
// with one token per CTA and 1.7 waves instead of two tokens per CTA and one
// wave, the CTA scheduler gives the SMs that move rows fastest more of them
// (staged combine 73.0 -> 71.5 us on DS-V3, Large 503 -> 500 us).  The ring
// reduce stays at one wave: two took DS-V3 to 75.5 and skewed to 37.0 us.
#ifndef LLMOE_PUT_WAVES
#define LLMOE_PUT_WAVES 2
#endif
#ifndef LLMOE_PUT_BATCH
#define LLMOE_PUT_BATCH 4
#endif
// The staged put moves rows in steps of kPutBatch chunks: measured against 8,
// 4 took the staged combine from 81.4 to 78.2 us on DS-V3 (skewed 38.3 -> 37.1,
// many-small 15.3 -> 14.3); the unpack keeps steps of 8, where 4 was no faster.
constexpr int kPutBatch = LLMOE_PUT_BATCH;


// Payload quad from two consecutive aligned quads a, b when the payload starts
// `phase` words into a: words phase .. phase+3 of (a, b).
__device__ __forceinline__ uint4 unshift_words(const uint4& a, const uint4& b, int phase) {
  switch (phase) {
    case 0: return a;
    case 1: return make_uint4(a.y, a.z, a.w, b.x);
    case 2: return make_uint4(a.z, a.w, b.x, b.y);
    default: return make_uint4(a.w, b.x, b.y, b.z);
  }
}

// Put: entry (src, t, k) choosing expert e sends [t][y row] to rank src's
// combine_recv[e][t] (row e * T_max + t of its receive region).  One warp
// moves 32 quads of one entry's row per unit; rank src's flag words are
// written by the CTA of its last token block.
__global__ void __launch_bounds__(kThreads, 4) combine_put_kernel(Geometry g, const void* __restrict__ y,
                                                                  const int64_t* __restrict__ idx) {
  extern __shared__ __align__(128) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  const int TBK = g.TB * g.K;
  const uint4** s_src = reinterpret_cast<const uint4**>(s.slot + TBK + (g.E & 1));
  uintptr_t* s_dst = reinterpret_cast<uintptr_t*>(s_src + TBK);

  const int src = blockIdx.x / g.nblk, b = blockIdx.x % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const bool last = (b == g.nblk - 1);
  const int nblock = (t1 - t0) * g.K;
  const bool early = (g.flags & LLMOE_FLAG_INPUTS_READY) != 0;
  release_next_grid();
  if (!early) wait_prior_grid();

  route_hist(g, idx, src, t0, t1, s, threadIdx.x, blockDim.x);
  uint8_t* rbase = g.base + src * g.rank_stride + g.recv_off;
  for (int q = threadIdx.x; q < nblock; q += blockDim.x) {
    const int e = s.ent[q], sl = route_slot(g, s, q);
    const uint4* row = nullptr;
    uintptr_t d = 0;
    if (sl >= 0) {
      row = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(y) +
                                           ((uint64_t)e * g.R * g.T_max + (uint64_t)src * g.T_max + sl) * g.row_bytes);
      d = pack_dest(rbase + ((uint64_t)e * g.T_max + (t0 + q / g.K)) * g.msg);
    }
    s_src[q] = row;
    s_dst[q] = d;
  }
  __syncthreads();
  if (early) wait_prior_grid();
  clean_other_set(g);
  if (last) route_count_block(s, nblock);

  // one warp per entry: its expert row in steps of up to kPutBatch
  // chunks, every load of a step before its first store; lane 0's previous
  // quad is lane 31's quad of the chunk before (the header word t before
  // chunk 0)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q = warp; q < nblock; q += kThreads / 32) {
    const uint4* row = s_src[q];
    if (row == nullptr) continue;  // the whole warp: masked entry
    const uintptr_t d = s_dst[q];
    uint4 carry = make_uint4(0, 0, 0, (uint32_t)(t0 + q / g.K));
    for (int c = 0; c < g.nchunks; c += kPutBatch) {
      const int n = min(kPutBatch, g.nchunks - c);
      uint4 cur[kPutBatch];
#pragma unroll
      for (int i = 0; i < kPutBatch; ++i) {
        const int j = (c + i) * 32 + lane;
        cur[i] = (i < n && j < g.nq) ? ld_stream16(row + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kPutBatch; ++i) {
        if (i < n) {
          const int j = (c + i) * 32 + lane;
          uint4 prev = shfl_up16(cur[i]);
          if (lane == 0) prev = carry;
          if (j < g.nq) put_quad(d, j, g.nq, prev, cur[i]);
          carry = shfl_idx16(cur[i], 31);
        }
      }
    }
  }

  if (last) {
    __syncthreads();
    // rank src's word e = rows expert e returned to src
    int64_t* w = reinterpret_cast<int64_t*>(g.base + src * g.rank_stride + g.sig_off);
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) put_signal(g, w + e, s.hist[e]);
  }
}

// Reduce: out[src][t] from the payloads of combine_recv[e_k][t], ascending k.
// One warp per (token, 32-quad chunk); the messages sit at 4-byte phases, so
// each lane loads its aligned quad, takes the next one from its neighbour and
// shifts the payload words into place.
// Payload quad j of a message whose payload starts `phase` 32-bit words past
// a 16-byte boundary, read with the widest loads that alignment allows (one
// 16-byte, two 8-byte or four 4-byte loads).  The phase is the same for the
// whole warp, so the branch does not diverge.
__device__ __forceinline__ uint4 ld_payload_quad(const uint8_t* pay, int phase, int j) {
  const uint8_t* p = pay + 16 * (size_t)j;
  if (phase == 0) return __ldg(reinterpret_cast<const uint4*>(p));
  if (phase == 2) {
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(p)), hi = __ldg(reinterpret_cast<const uint2*>(p + 8));
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
  return make_uint4(__ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3));
}

// Reduce through a shared-memory ring (combine_reduce_ring_kernel), for grids
// with more than one unit per consumer warp.  A CTA takes a contiguous range of the
// R * T * nchunks (token, 512 B chunk) units.  Its producer warp copies each
// unit's K message chunks into one ring stage with cp.async.bulk, lane k the
// chunk of entry k: the 16-byte-aligned span that covers the chunk (the
// payload sits at a 4-byte phase, so one quad more when the phase is not
// zero).  Consumer warp w takes the units at ring positions w, w + C, ...:
// lane j reads quads j and j + 1 of each entry's span from shared memory,
// shifts the payload words into place and accumulates them, ascending k.
// The copies need no registers while in flight, so a CTA keeps kRedStages
// units' messages in flight, where register loads held four.
#ifndef LLMOE_RED_STAGES
#define LLMOE_RED_STAGES 4
#endif
#ifndef LLMOE_RED_CONSUMERS
#define LLMOE_RED_CONSUMERS 2
#endif
#ifndef LLMOE_RED_WIDTH
#define LLMOE_RED_WIDTH 1
#endif
constexpr int kRedStages = LLMOE_RED_STAGES;
constexpr int kRedConsumers = LLMOE_RED_CONSUMERS;
constexpr int kRedThreads = 32 * (1 + kRedConsumers);
constexpr int kRedWidth = LLMOE_RED_WIDTH;  // 512 B chunks per unit
constexpr int kRedSlot = (32 * kRedWidth + 1) * 16;  // one entry's span: the unit's payload quads and the one the phase spills into
// Stage s is used only by consumer warp s % kRedConsumers, so a consumer's
// parity waits on a stage follow each other in order; with a stage shared by
// two consumers, one could wait for a phase two ahead of the barrier's and
// take the parity of an old phase for its own.
static_assert(kRedStages % kRedConsumers == 0, "every ring stage belongs to one consumer warp");

struct RedMeta {
  int phase;  // the payload's 4-byte phase; -1: masked entry
  float w;
};

template <int DT>
__global__ void __launch_bounds__(kRedThreads) combine_reduce_ring_kernel(Geometry g, const int64_t* __restrict__ idx,
                                                                          const float* __restrict__ topk_w,
                                                                          void* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int K = g.K;
  uint8_t* data = smem;  // [stage][k][kRedSlot]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kRedStages * K * kRedSlot);
  uint64_t* empty = full + kRedStages;
  RedMeta* meta = reinterpret_cast<RedMeta*>(empty + kRedStages);  // [stage][k]
  int64_t* unit_tok = reinterpret_cast<int64_t*>(meta + kRedStages * K);  // [stage]
  __shared__ int s_stop[kRedConsumers];  // per consumer warp: the first position it did not consume
  __shared__ int s_issued;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRedStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init_fence();
    s_issued = 0;
  }
  release_next_grid();
  wait_prior_grid();
  __syncthreads();
  const int nu = (g.nchunks + kRedWidth - 1) / kRedWidth;  // units per token
  const int64_t nunits = (int64_t)g.R * g.T * nu;
  const int64_t ubeg = nunits * blockIdx.x / gridDim.x, uend = nunits * (blockIdx.x + 1) / gridDim.x;
  const int npos = (int)(uend - ubeg);

  if (warp == 0) {
    // producer: lanes k < K hold entry k's expert id and weight of the current token
    int64_t tok = ubeg / nu;
    int c = (int)(ubeg - tok * nu);
    int src = (int)(tok / g.T), t = (int)(tok - (int64_t)src * g.T);
    long long e_lane = -1;
    float w_lane = 0.0f;
    bool fresh = true, ok = true;
    int pos = 0;
    for (; pos < npos; ++pos) {
      if (fresh) {
        e_lane = -1;
        w_lane = 0.0f;
        if (lane < K) {
          e_lane = idx[tok * K + lane];
          w_lane = topk_w[tok * K + lane];
        }
        fresh = false;
      }
      const int sidx = pos % kRedStages, use = pos / kRedStages;
      if (lane == 0 && use > 0) ok = mbar_wait(&empty[sidx], (use - 1) & 1, g.err);
      ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
      if (!ok) break;
      const int len = min(512 * kRedWidth, g.row_bytes - 512 * kRedWidth * c);
      const bool valid = lane < K && e_lane >= 0 && e_lane < g.E;
      uint32_t bytes = 0;
      int phase = -1;
      const uint8_t* span = nullptr;
      if (valid) {
        const uint8_t* msg = g.base + src * g.rank_stride + g.recv_off + ((uint64_t)e_lane * g.T_max + t) * g.msg;
        const uint8_t* p = msg + 4 + 512 * kRedWidth * (size_t)c;
        phase = (int)((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
        span = p - 4 * phase;
        bytes = (uint32_t)len + (phase != 0 ? 16u : 0u);
        if (g.err != nullptr && c == 0 && *reinterpret_cast<const int32_t*>(msg) != t)
          report(g.err, LLMOE_DEV_BAD_MESSAGE);
      }
      if (lane < K) meta[sidx * K + lane] = RedMeta{phase, w_lane};
      if (lane == 0) unit_tok[sidx] = tok;
      uint32_t total = bytes;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[sidx], total);
      __syncwarp();
      if (valid) bulk_load(data + ((size_t)sidx * K + lane) * kRedSlot, span, bytes, &full[sidx]);
      if (++c == nu) {
        c = 0;
        ++tok;
        if (++t == g.T) {
          t = 0;
          ++src;
        }
        fresh = true;
      }
    }
    if (lane == 0) s_issued = pos;
    __syncwarp();
  } else {
    const int cw = warp - 1;
    int pos = cw;
    for (; pos < npos; pos += kRedConsumers) {
      const int sidx = pos % kRedStages;
      if (!mbar_wait(&full[sidx], (pos / kRedStages) & 1, g.err)) break;
      const int64_t tok = unit_tok[sidx];
      const int c = (int)((ubeg + pos) - tok * nu);
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) + tok * g.row_bytes);
#pragma unroll
      for (int i = 0; i < kRedWidth; ++i) {
        const int j = (c * kRedWidth + i) * 32 + lane;
        if (j >= g.nq) break;
        float acc[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) acc[a] = 0.0f;
        const uint4* q = reinterpret_cast<const uint4*>(data + (size_t)sidx * K * kRedSlot) + 32 * i + lane;
        for (int k = 0; k < K; ++k, q += kRedSlot / 16) {  // ascending k
          const RedMeta m = meta[sidx * K + k];
          if (m.phase >= 0) axpy_q<DT>(acc, m.w, unshift_words(q[0], q[1], m.phase));
        }
        orow[j] = pack_q<DT>(acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sidx]);
    }
    if (lane == 0) s_stop[cw] = pos;
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // after a timeout: wait (bounded) for the copies nobody consumed
    for (int p = max(0, s_issued - kRedStages); p < s_issued; ++p)
      if (p >= s_stop[p % kRedConsumers] && !mbar_wait(&full[p % kRedStages], (p / kRedStages) & 1, g.err)) break;
  }
}

size_t reduce_smem_bytes(const Geometry& g) {
  return (size_t)kRedStages * g.K * kRedSlot + 2 * kRedStages * sizeof(uint64_t) +
         (size_t)kRedStages * g.K * sizeof(RedMeta) + kRedStages * sizeof(int64_t);
}

// Reduce with register loads (combine_reduce_kernel), for smaller grids:
// there a unit's latency is the kernel's, and the ring's producer hand-off
// adds to it (many-small staged combine 14.4 us this way, 16.3 us through the
// ring).
#ifndef LLMOE_REDUCE_KBATCH
#define LLMOE_REDUCE_KBATCH 4
#endif
constexpr int kReduceBatch = LLMOE_REDUCE_KBATCH;  // messages whose loads a warp has in flight at once

// Each warp takes a contiguous range of the R * T * nchunks (token, chunk)
// units, so it meets a new token once per nchunks units at most: lanes k < K
// then load that token's expert id and weight (one memory round trip), and
// every unit of the token reuses them from registers.
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) combine_reduce_kernel(Geometry g, const int64_t* __restrict__ idx,
                                                                     const float* __restrict__ topk_w,
                                                                     void* __restrict__ out) {
  release_next_grid();
  wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t nunits = (int64_t)g.R * g.T * g.nchunks;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t ubeg = nunits * gw / nwarps, uend = nunits * (gw + 1) / nwarps;
  if (ubeg >= uend) return;
  int64_t tok = ubeg / g.nchunks;  // walked forward unit by unit from here
  int c = (int)(ubeg - tok * g.nchunks);
  int src = (int)(tok / g.T), t = (int)(tok - (int64_t)src * g.T);
  bool fresh = true;
  long long e_lane = -1;
  float w_lane = 0.0f;
  for (int64_t left = uend - ubeg; left > 0; --left) {
    if (fresh) {  // the whole warp: lane k holds entry k of the token
      e_lane = -1;
      w_lane = 0.0f;
      if (lane < g.K) {
        e_lane = idx[tok * g.K + lane];
        w_lane = topk_w[tok * g.K + lane];
      }
      fresh = false;
    }
    const int j = c * 32 + lane;
    const uint8_t* rbase = g.base + src * g.rank_stride + g.recv_off;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int k0 = 0; k0 < g.K; k0 += kReduceBatch) {
      // the batch's messages: lane j reads payload quad j at the message's
      // own alignment
      uint4 a[kReduceBatch];
      const uint8_t* msg[kReduceBatch];
      float wk[kReduceBatch];
#pragma unroll
      for (int i = 0; i < kReduceBatch; ++i) {
        const int k = k0 + i;
        const long long e = __shfl_sync(0xffffffffu, e_lane, k & 31);
        wk[i] = __shfl_sync(0xffffffffu, w_lane, k & 31);
        a[i] = make_uint4(0, 0, 0, 0);
        msg[i] = nullptr;
        if (k < g.K && e >= 0 && e < g.E) {  // the whole warp
          msg[i] = rbase + ((uint64_t)e * g.T_max + t) * g.msg;
          const int phase = (int)(((reinterpret_cast<uintptr_t>(msg[i]) + 4) >> 2) & 3);
          if (j < g.nq) a[i] = ld_payload_quad(msg[i] + 4, phase, j);
        }
      }
#pragma unroll
      for (int i = 0; i < kReduceBatch; ++i) {  // ascending k
        if (msg[i] == nullptr) continue;
        if (g.err != nullptr && j == 0 && *reinterpret_cast<const int32_t*>(msg[i]) != t)
          report(g.err, LLMOE_DEV_BAD_MESSAGE);
        if (j < g.nq) axpy_q<DT>(acc, wk[i], a[i]);
      }
    }
    if (j < g.nq)
      reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) + ((int64_t)src * g.T + t) * g.row_bytes)[j] =
          pack_q<DT>(acc);
    if (++c == g.nchunks) {  // the next token
      c = 0;
      ++tok;
      if (++t == g.T) {
        t = 0;
        ++src;
      }
      fresh = true;
    }
  }
}


// ---------------------------------------------------------------------------
// unpack, and the dispatch whose CTAs signal each other
// ---------------------------------------------------------------------------

// Unpack after a dispatch, balanced over the grid: every CTA reads all E * R
// bucket counts and their exclusive prefix (shared memory), so the N received
// rows x chunks split evenly over all warps whatever the routing's skew.  A
// warp finds the bucket of its first row by binary search and then walks its
// range row by row (unpack_row).
constexpr int kMaxScanBuckets = 8192;
#ifndef LLMOE_UNPACK_THREADS
#define LLMOE_UNPACK_THREADS 512
#endif
// Threads of a balanced-unpack CTA: every CTA reads and scans all the count
// words, so fewer, larger CTAs read them fewer times for the same warps.
constexpr int kUnpackThreads = LLMOE_UNPACK_THREADS;
constexpr int kCountLoads = 8;  // count words a thread has in flight in the prologue

__device__ __forceinline__ int find_bucket(const int* pre, int nb, int r) {
  int lo = 0, hi = nb - 1;  // largest b with pre[b] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}


// Moves chunks [c, cend) of one received message's payload to its row of the
// experts' input: up to kRowBatch consecutive chunks per step, every load of
// the step issued before the first store.
// - Through L1 (kL2Only false): lane j reads payload quad j at the message's
//   own alignment (ld_payload_quad); the narrower loads of one quad hit the
//   lines its first load brought into L1.
// - L2 only (kL2Only true: the message may have been written by a CTA of the
//   same launch, so no L1 copy may be used): every aligned quad is loaded
//   once, and lane j rebuilds its quad from its own aligned quad and the next,
//   which comes from the next lane (shfl_down) or, for lane 31, from lane 0 of
//   the next chunk.  Narrow loads there would fetch each quad's sectors from
//   L2 up to four times.
template <bool kL2Only>
__device__ __forceinline__ void unpack_row(const Geometry& g, const uint8_t* msg, uint4* __restrict__ drow, int c,
                                           int cend, int lane) {
  const uint8_t* pay = msg + 4;
  const int phase = (int)((reinterpret_cast<uintptr_t>(pay) >> 2) & 3);
  if constexpr (!kL2Only) {
    for (; c < cend; c += kRowBatch) {
      const int n = min(kRowBatch, cend - c);
      uint4 a[kRowBatch];
#pragma unroll
      for (int i = 0; i < kRowBatch; ++i) {
        const int j = (c + i) * 32 + lane;
        a[i] = make_uint4(0, 0, 0, 0);
        if (i < n && j < g.nq) a[i] = ld_payload_quad(pay, phase, j);
      }
#pragma unroll
      for (int i = 0; i < kRowBatch; ++i) {
        const int j = (c + i) * 32 + lane;
        if (i < n && j < g.nq) drow[j] = a[i];
      }
    }
  } else {
    const uint4* qb = reinterpret_cast<const uint4*>(reinterpret_cast<uintptr_t>(pay) & ~(uintptr_t)15);
    for (; c < cend; c += kRowBatch) {
      const int n = min(kRowBatch, cend - c);
      uint4 a[kRowBatch];
#pragma unroll
      for (int i = 0; i < kRowBatch; ++i) {
        const int j = (c + i) * 32 + lane;
        a[i] = make_uint4(0, 0, 0, 0);
        if (i < n && (j < g.nq || (j == g.nq && phase != 0))) a[i] = __ldcg(qb + j);
      }
      // lane 31 of the step's last chunk: the quad after it, unless past the payload
      const int jl = (c + n - 1) * 32 + 31;
      uint4 tail = make_uint4(0, 0, 0, 0);
      if (lane == 31 && phase != 0 && jl < g.nq) tail = __ldcg(qb + jl + 1);
#pragma unroll
      for (int i = 0; i < kRowBatch; ++i) {
        if (i < n) {
          const int j = (c + i) * 32 + lane;
          uint4 q = a[i];
          if (phase != 0) {
            uint4 bq = shfl_down16(a[i]);
            uint4 nx = tail;
            if (i + 1 < kRowBatch) {
              const uint4 t = shfl_idx16(a[min(i + 1, kRowBatch - 1)], 0);
              if (i + 1 < n) nx = t;
            }
            if (lane == 31) bq = nx;
            q = unshift_words(a[i], bq, phase);
          }
          if (j < g.nq) drow[j] = q;
        }
      }
    }
  }
}

__global__ void
__launch_bounds__(kUnpackThreads, kUnpackThreads >= 1024 ? 1 : LLMOE_UNPACK_MIN_BLOCKS * 256 / kUnpackThreads)
    unpack_balanced_kernel(Geometry g, void* __restrict__ recv_x, int32_t* __restrict__ recv_src) {
  __shared__ int s_pre[kMaxScanBuckets];
  __shared__ int s_part[kUnpackThreads / 32];
  release_next_grid();
  wait_prior_grid();
  const int nb = g.E * g.R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int b0 = 0; b0 < nb; b0 += kCountLoads * kUnpackThreads) {
    int64_t c[kCountLoads];
#pragma unroll
    for (int i = 0; i < kCountLoads; ++i) {
      const int b = b0 + i * kUnpackThreads + tid, e = b / g.R, src = b - e * g.R;
      c[i] = b < nb ? reinterpret_cast<const int64_t*>(g.base + (e / g.L) * g.rank_stride + g.sig_off)
                          [(int64_t)(e % g.L) * g.R + src]
                    : 0;
    }
#pragma unroll
    for (int i = 0; i < kCountLoads; ++i) {
      const int b = b0 + i * kUnpackThreads + tid;
      if (b < nb) s_pre[b] = (int)max((int64_t)0, min(c[i], (int64_t)g.T_max));
    }
  }
  __syncthreads();
  // exclusive prefix: each thread scans a contiguous segment, the segment
  // totals are scanned across the block
  const int seg = (nb + kUnpackThreads - 1) / kUnpackThreads, lo = min(nb, tid * seg), hi = min(nb, lo + seg);
  int sum = 0;
  for (int b = lo; b < hi; ++b) sum += s_pre[b];
  int incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s_part[warp] = incl;
  __syncthreads();
  int warp_base = 0;
  for (int w = 0; w < warp; ++w) warp_base += s_part[w];
  int total = 0;
  for (int w = 0; w < kUnpackThreads / 32; ++w) total += s_part[w];
  int run = warp_base + incl - sum;
  __syncthreads();  // every segment read its counts before any is overwritten
  for (int b = lo; b < hi; ++b) {
    const int cb = s_pre[b];
    s_pre[b] = run;
    run += cb;
  }
  __syncthreads();

  // the warp's contiguous range [ubeg, uend) of (row, chunk) units
  const int64_t nunits = (int64_t)total * g.nchunks;
  const int64_t nwarps = ((int64_t)gridDim.x * kUnpackThreads) >> 5;
  const int64_t gw = ((int64_t)blockIdx.x * kUnpackThreads + tid) >> 5;
  const int64_t per = (nunits + nwarps - 1) / nwarps;
  const int64_t ubeg = min(nunits, gw * per), uend = min(nunits, ubeg + per);
  if (ubeg >= uend) return;
  int r = (int)(ubeg / g.nchunks);
  int c = (int)(ubeg - (int64_t)r * g.nchunks);
  int64_t left = uend - ubeg;
  int bucket = find_bucket(s_pre, nb, r);
  while (left > 0) {
    while (bucket + 1 < nb && s_pre[bucket + 1] <= r) ++bucket;  // rows only grow along the range
    const int slot = r - s_pre[bucket];
    const int e = bucket / g.R, src = bucket - e * g.R, le = e % g.L;
    const uint8_t* msg = g.base + (e / g.L) * g.rank_stride + g.recv_off +
                         (((uint64_t)le * g.R + src) * g.T_max + slot) * g.msg;
    const int64_t orow = (int64_t)bucket * g.T_max + slot;
    uint4* drow = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(recv_x) + orow * g.row_bytes);
    const int cend = (int)min((int64_t)g.nchunks, c + left);  // this row's chunks in the range
    const bool head = (c == 0);
    int hv = 0;
    if (head && lane == 0) hv = *reinterpret_cast<const int32_t*>(msg);
    left -= cend - c;
    unpack_row<false>(g, msg, drow, c, cend, lane);
    if (head && lane == 0) recv_src[orow] = hv;
    c = 0;
    ++r;
  }
}

// Unpack after a dispatch with at least as many buckets as routed entries
// (few rows per bucket, so little skew to balance), or more buckets than the
// balanced kernel's shared prefix holds: one warp per bucket (expert e,
// source src), grid-stride; the bucket's count word gives how many of its
// slots hold a message, and the warp unpacks them row by row.
__global__ void __launch_bounds__(kThreads, LLMOE_UNPACK_MIN_BLOCKS)
    unpack_kernel(Geometry g, void* __restrict__ recv_x, int32_t* __restrict__ recv_src) {
  release_next_grid();
  wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int nbuckets = g.E * g.R;  // E <= LLMOE_MAX_EXPERTS and R <= E: fits an int
  const int nwarps = (gridDim.x * kThreads) >> 5;
  for (int bucket = (blockIdx.x * kThreads + threadIdx.x) >> 5; bucket < nbuckets; bucket += nwarps) {
    const int e = bucket / g.R, src = bucket - e * g.R, dst = e / g.L, le = e % g.L;
    const uint8_t* rank = g.base + dst * g.rank_stride;
    const int64_t c64 = reinterpret_cast<const int64_t*>(rank + g.sig_off)[(int64_t)le * g.R + src];
    const int cnt = (int)max((int64_t)0, min(c64, (int64_t)g.T_max));
    const uint8_t* msg0 = rank + g.recv_off + ((uint64_t)le * g.R + src) * g.T_max * g.msg;
    uint8_t* row0 = reinterpret_cast<uint8_t*>(recv_x) + (int64_t)bucket * g.T_max * g.row_bytes;
    for (int slot = 0; slot < cnt; ++slot) {
      const uint8_t* msg = msg0 + (size_t)slot * g.msg;
      int hv = 0;
      if (lane == 0) hv = *reinterpret_cast<const int32_t*>(msg);
      unpack_row<false>(g, msg, reinterpret_cast<uint4*>(row0 + (size_t)slot * g.row_bytes), 0, g.nchunks, lane);
      if (lane == 0) recv_src[(int64_t)bucket * g.T_max + slot] = hv;
    }
  }
}

__device__ __forceinline__ long long ld_acquire_gpu(const long long* p) {
  long long v;
  asm volatile("ld.acquire.gpu.global.s64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(long long* p, long long v) {
  asm volatile("st.release.gpu.global.s64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Rank e / L's signal word le * R + src: the recv count of bucket (e, src).
__device__ __forceinline__ long long* signal_word(const Geometry& g, int e, int src) {
  return reinterpret_cast<long long*>(g.base + (e / g.L) * g.rank_stride + g.sig_off) + ((int64_t)(e % g.L) * g.R + src);
}

// Consumer work of the signalled dispatch for source rank s by this CTA,
// member k of the Gs CTAs serving s.  The CTA's threads wait (bounded) for
// s's signal words in parallel, scan the counts into s_pre (E ints of shared
// memory) and split s's received (row, chunk) units evenly over the Gs * 8
// warps.  Returns early, after reporting LLMOE_DEV_TIMEOUT, when a word of s
// is not raised within the spin limit.  Called by every thread of the CTA.
__device__ void consume_source(const Geometry& g, int s, int k, int Gs, int* s_pre, int* s_part, int* s_ok,
                               void* __restrict__ recv_x, int32_t* __restrict__ recv_src, long long spin_limit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();  // s_pre / s_ok of the previous use have been read
  if (tid == 0) *s_ok = 1;
  __syncthreads();
  for (int e = tid; e < g.E; e += kThreads) {
    const long long* w = signal_word(g, e, s);
    long long v = ld_acquire_gpu(w);
    const long long start = clock64();
    while (v == 0 && clock64() - start <= spin_limit) {
      __nanosleep(64);
      v = ld_acquire_gpu(w);
    }
    s_pre[e] = v < 0 ? (int)min(-v - 1, (long long)g.T_max) : 0;
    if (v >= 0) *s_ok = 0;  // never raised (or not a raised signal)
  }
  __syncthreads();  // every count, and every thread's acquire, before any read of s's rows
  if (*s_ok == 0) {
    if (tid == 0) report(g.err, LLMOE_DEV_TIMEOUT);
    return;
  }
  // exclusive prefix of the counts (each thread a contiguous segment)
  const int seg = (g.E + kThreads - 1) / kThreads, lo = min(g.E, tid * seg), hi = min(g.E, lo + seg);
  int sum = 0;
  for (int e = lo; e < hi; ++e) sum += s_pre[e];
  int incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s_part[warp] = incl;
  __syncthreads();
  int run = incl - sum, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) run += s_part[w];
    total += s_part[w];
  }
  __syncthreads();  // every segment read its counts before any is overwritten
  for (int e = lo; e < hi; ++e) {
    const int ce = s_pre[e];
    s_pre[e] = run;
    run += ce;
  }
  __syncthreads();

  // this warp's range [ubeg, uend) of s's (row, chunk) units
  const int64_t nunits = (int64_t)total * g.nchunks;
  const int64_t ws = (int64_t)Gs * (kThreads / 32), wi = (int64_t)k * (kThreads / 32) + warp;
  const int64_t per = (nunits + ws - 1) / ws;
  const int64_t ubeg = min(nunits, wi * per), uend = min(nunits, ubeg + per);
  if (ubeg >= uend) return;
  int r = (int)(ubeg / g.nchunks);
  int c = (int)(ubeg - (int64_t)r * g.nchunks);
  int64_t left = uend - ubeg;
  int e = find_bucket(s_pre, g.E, r);
  auto end_of = [&](int ex) { return ex + 1 < g.E ? s_pre[ex + 1] : total; };
  int slot = r - s_pre[e];
  while (left > 0) {
    while (slot >= end_of(e) - s_pre[e]) {  // past this expert's rows: the next expert with rows
      slot = 0;
      ++e;
    }
    const int le = e % g.L;
    const uint8_t* msg = g.base + (e / g.L) * g.rank_stride + g.recv_off +
                         (((uint64_t)le * g.R + s) * g.T_max + slot) * g.msg;
    const int64_t orow = ((int64_t)e * g.R + s) * g.T_max + slot;
    const int cend = (int)min((int64_t)g.nchunks, c + left);  // this row's chunks in the range
    const bool head = (c == 0);
    int hv = 0;
    if (head && lane == 0) hv = __ldcg(reinterpret_cast<const int32_t*>(msg));
    left -= cend - c;
    unpack_row<true>(g, msg, reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(recv_x) + orow * g.row_bytes), c,
                     cend, lane);
    if (head && lane == 0) recv_src[orow] = hv;
    c = 0;
    ++slot;
  }
}

// Cooperative: every CTA is resident, so a consumer that waits on a signal
// word only waits for producers that are running.  Producer work (CTA =
// source rank src, token block) is the dispatch; the CTA that completes a
// source (per-source counter in `done`) raises its signal words as
// -(count + 1).  Consumer work takes buckets (expert e, source src) round
// robin, waits (bounded) for the bucket's word, unpacks its rows and rewrites
// the word to the plain count.
__global__ void __launch_bounds__(kThreads, 3) dispatch_signaled_kernel(Geometry g, const void* __restrict__ x,
                                                                        const int64_t* __restrict__ idx,
                                                                        void* __restrict__ recv_x,
                                                                        int32_t* __restrict__ recv_src,
                                                                        int32_t* __restrict__ done, long long spin_limit) {
  extern __shared__ __align__(128) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  uintptr_t* s_dst = reinterpret_cast<uintptr_t*>(s.slot + g.TB * g.K + (g.E & 1));
  __shared__ int s_last;

  const int src = blockIdx.x / g.nblk, b = blockIdx.x % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const int nblock = (t1 - t0) * g.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- producer: this CTA's rows
  route_hist(g, idx, src, t0, t1, s, threadIdx.x, blockDim.x);
  for (int q = threadIdx.x; q < nblock; q += blockDim.x) {
    const int e = s.ent[q], sl = route_slot(g, s, q);
    uintptr_t d = 0;
    if (sl >= 0) {
      const int dst = e / g.L, le = e % g.L;
      const uint64_t row = ((uint64_t)le * g.R + src) * g.T_max + sl;
      d = pack_dest(g.base + dst * g.rank_stride + g.recv_off + row * g.msg);
    }
    s_dst[q] = d;
  }
  __syncthreads();
  const int nunits = (t1 - t0) * g.nchunks;
  for (int u = warp; u < nunits; u += kThreads / 32) {
    const int tl = u / g.nchunks, c = u % g.nchunks, t = t0 + tl, j = c * 32 + lane;
    const uint4* xrow =
        reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(x) + ((int64_t)src * g.T + t) * g.row_bytes);
    const uint4 cur = j < g.nq ? __ldg(xrow + j) : make_uint4(0, 0, 0, 0);
    uint4 prev = shfl_up16(cur);
    if (lane == 0) prev = j == 0 ? make_uint4(0, 0, 0, (uint32_t)t) : __ldg(xrow + j - 1);
    if (j < g.nq)
      for (int k = 0; k < g.K; ++k) {
        const uintptr_t d = s_dst[tl * g.K + k];
        if (d != 0) put_quad(d, j, g.nq, prev, cur);
      }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's rows before its completion count
    s_last = atomicAdd(&done[src], 1) == g.nblk - 1;
  }
  __syncthreads();
  if (s_last) {
    // every CTA of src has written its rows: raise src's signal words
    __threadfence();
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) s.hist[e] = 0;
    __syncthreads();
    const int64_t* src_idx = idx + (int64_t)src * g.T * g.K;
    for (int i = threadIdx.x; i < g.T * g.K; i += blockDim.x) {
      const int64_t e = src_idx[i];
      if (e >= 0 && e < g.E) atomicAdd(&s.hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      long long* w = reinterpret_cast<long long*>(g.base + (e / g.L) * g.rank_stride + g.sig_off) +
                     ((int64_t)(e % g.L) * g.R + src);
      if (g.err != nullptr && *reinterpret_cast<volatile long long*>(w) != 0) report(g.err, LLMOE_DEV_STALE_SIGNAL);
      st_release_gpu(w, -(long long)s.hist[e] - 1);
    }
    if (threadIdx.x == 0) done[src] = 0;  // ready for the next call
  }

  // ---- consumer: CTAs grouped by source rank (consume_source).  Consumers
  // do not rewrite the words: the last CTA to finish turns every raised word
  // back into its plain count.
  __shared__ int s_part[kThreads / 32];
  __shared__ int s_ok;
  if ((int)gridDim.x >= g.R) {
    const int sg = blockIdx.x % g.R;
    consume_source(g, sg, blockIdx.x / g.R, ((int)gridDim.x - sg + g.R - 1) / g.R, s.hist, s_part, &s_ok, recv_x,
                   recv_src, spin_limit);
  } else {
    for (int sg = blockIdx.x; sg < g.R; sg += gridDim.x)
      consume_source(g, sg, 0, 1, s.hist, s_part, &s_ok, recv_x, recv_src, spin_limit);
  }
  __syncthreads();  // the CTA's consumers are done
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's reads of the signal words before its completion count
    s_last = atomicAdd(&done[g.R], 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    constexpr int kBatch = 8;  // words a thread has in flight at once
    const int nw = g.E * g.R;
    for (int i0 = 0; i0 < nw; i0 += kThreads * kBatch) {
      long long* w[kBatch];
      long long v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * kThreads + threadIdx.x;
        w[j] = nullptr;
        v[j] = 0;
        if (i < nw) {
          const int e = i / g.R;
          w[j] = signal_word(g, e, i - e * g.R);
          v[j] = __ldcg(w[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (v[j] < 0) *w[j] = -v[j] - 1;  // the plain count, as a dispatch leaves it
    }
    if (threadIdx.x == 0) done[g.R] = 0;  // ready for the next call
  }
}

__global__ void __launch_bounds__(kThreads) route_kernel(Geometry g, const int64_t* __restrict__ idx,
                                                         int32_t* __restrict__ slot_out,
                                                         int64_t* __restrict__ counts) {
  extern __shared__ __align__(128) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  const int src = blockIdx.x / g.nblk, b = blockIdx.x % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const bool last = (b == g.nblk - 1);
  release_next_grid();
  wait_prior_grid();
  route_hist(g, idx, src, t0, t1, s, threadIdx.x, blockDim.x);
  const int nblock = (t1 - t0) * g.K;
  for (int q = threadIdx.x; q < nblock; q += blockDim.x)
    slot_out[((int64_t)src * g.T + t0) * g.K + q] = route_slot(g, s, q);
  if (last) {
    __syncthreads();
    route_count_block(s, nblock);
    __syncthreads();
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) counts[(int64_t)e * g.R + src] = s.hist[e];
  }
}

__global__ void __launch_bounds__(kThreads) clean_kernel(uint8_t* base, uint64_t rank_stride, uint64_t sig_off,
                                                         int R, int E) {
  const int64_t n = (int64_t)R * E;
  release_next_grid();
  wait_prior_grid();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / E, e = i % E;
    reinterpret_cast<int64_t*>(base + r * rank_stride + sig_off)[e] = 0;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

bool mul_u64(uint64_t a, uint64_t b, uint64_t* r) { return !__builtin_mul_overflow(a, b, r); }
bool add_u64(uint64_t a, uint64_t b, uint64_t* r) { return !__builtin_add_overflow(a, b, r); }

struct LayoutInfo {
  uint64_t total, msg, send, recv, sig;
};

// LLMoEBufferLayout<T>: send = max(T*msg, E*T*msg), recv = E*T*msg (both
// roles), sig = 8*E; each region twice; msg = sizeof(int) + hidden*sizeof(T).
bool layout_info(int T, int H, int R, int E, int es, LayoutInfo* out) {
  if (T < 1 || H < 1 || R < 1 || E < 1 || es < 1) return false;
  uint64_t msg, et, dsend, csend, recv, total = 0, two;
  if (!mul_u64((uint64_t)H, (uint64_t)es, &msg) || !add_u64(msg, 4, &msg)) return false;
  if (!mul_u64((uint64_t)T, msg, &dsend)) return false;
  if (!mul_u64((uint64_t)E, (uint64_t)T, &et) || !mul_u64(et, msg, &csend)) return false;
  const uint64_t send = dsend > csend ? dsend : csend;
  recv = csend;  // dispatch and combine receive regions both hold E*T messages
  if (send % 4 != 0 || recv % 4 != 0) return false;
  const uint64_t sig = (uint64_t)E * 8;
  if (!mul_u64(send, 2, &two) || !add_u64(total, two, &total)) return false;
  if (!mul_u64(recv, 2, &two) || !add_u64(total, two, &total)) return false;
  if (!add_u64(total, 2 * sig, &total)) return false;
  *out = LayoutInfo{total, msg, send, recv, sig};
  return true;
}

int dtype_size(int dtype) {
  switch (dtype) {
    case LLMOE_DTYPE_BF16: return 2;
    case LLMOE_DTYPE_FP16: return 2;
    case LLMOE_DTYPE_FP32: return 4;
    default: return 0;
  }
}

// Per-device caches of device queries.  Host threads may call the library
// concurrently: every entry is an atomic, and two threads that miss together
// both query and store the same value.
constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < kMaxDevices) {
    const int c = g_num_sms[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < kMaxDevices) g_num_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validates a buffer set and fills the launch geometry.  need_buffers: the
// call writes the rank buffers (base / rank_stride / set must be valid).
int make_geometry(const llmoe_buf_set_t* bs, bool need_buffers, Geometry* g) {
  if (bs == nullptr) return LLMOE_ERR_INVALID_ARGUMENT;
  const int T_max = bs->num_max_tokens, T = bs->num_tokens, H = bs->hidden, R = bs->num_ranks,
            E = bs->num_experts, K = bs->num_topk;
  const int es = dtype_size(bs->dtype);
  if (es == 0 || T_max < 1 || T < 0 || T > T_max || H < 1 || ((int64_t)H * es) % 16 != 0 || R < 1 || E < R ||
      E % R != 0 || E > LLMOE_MAX_EXPERTS || K < 1 || K > LLMOE_MAX_TOPK || K > E)
    return LLMOE_ERR_INVALID_ARGUMENT;
  const int set = need_buffers ? bs->set : 0;
  if (set != 0 && set != 1) return LLMOE_ERR_INVALID_ARGUMENT;
  if (bs->err != nullptr && !aligned(bs->err, 4)) return LLMOE_ERR_INVALID_ARGUMENT;
  LayoutInfo li;
  if (!layout_info(T_max, H, R, E, es, &li)) return LLMOE_ERR_INVALID_ARGUMENT;
  // every index the kernels form stays below 2^63
  uint64_t rows, bytes;
  if (!mul_u64((uint64_t)E * (uint64_t)R, (uint64_t)T_max, &rows) || !mul_u64(rows, (uint64_t)H * es, &bytes) ||
      bytes > (uint64_t)INT64_MAX / 2)
    return LLMOE_ERR_INVALID_ARGUMENT;
  if (need_buffers) {
    uint64_t span;
    if (bs->base == nullptr || !aligned(bs->base, 16) || bs->rank_stride % 16 != 0 || bs->rank_stride < li.total ||
        !mul_u64(bs->rank_stride, (uint64_t)R, &span))
      return LLMOE_ERR_INVALID_ARGUMENT;
  }
  g->base = static_cast<uint8_t*>(bs->base);
  g->rank_stride = bs->rank_stride;
  g->recv_off = 2 * li.send + li.recv * (uint64_t)set;
  g->sig_off = 2 * li.send + 2 * li.recv + li.sig * (uint64_t)set;
  g->other_sig_off = 2 * li.send + 2 * li.recv + li.sig * (uint64_t)(set ^ 1);
  g->msg = li.msg;
  g->err = bs->err;
  g->flags = bs->flags;
  g->T_max = T_max;
  g->T = T;
  g->H = H;
  g->R = R;
  g->E = E;
  g->K = K;
  g->L = E / R;
  // e / L as a multiply-high: exact for e < 2^16 because e * (L_mul * L - 2^32) < 2^32
  g->L_mul = g->L == 1 ? 0u : (uint32_t)(((1ull << 32) + g->L - 1) / g->L);
  g->dtype = bs->dtype;
  g->row_bytes = H * es;
  g->nq = g->row_bytes / 16;
  g->nchunks = (g->nq + 31) / 32;
  g->TB = 1;
  g->nblk = T > 0 ? T : 1;
  g->dsplit = 1;
  g->csplit = 1;
  g->pf_units = 1;
  return LLMOE_SUCCESS;
}

// Tokens per CTA: the fewest that keep the grid (plus extra_ctas other CTAs)
// within one wave of resident CTAs (SMs x blocks_per_sm), at most
// kMaxTokensPerBlock.
void set_blocking(Geometry* g, int blocks_per_sm, int extra_ctas = 0) {
  const int64_t tokens = (int64_t)g->R * g->T;
  int64_t wave = (int64_t)num_sms() * (blocks_per_sm > 0 ? blocks_per_sm : 1) - extra_ctas;
  if (wave < 1) wave = 1;
  int64_t tb = (tokens + wave - 1) / wave;
  if (tb < 1) tb = 1;
  if (tb > kMaxTokensPerBlock) tb = kMaxTokensPerBlock;
  g->TB = (int)tb;
  g->nblk = g->T > 0 ? (g->T + g->TB - 1) / g->TB : 1;
}

constexpr int kMaxSlots = 44;  // kslot values: kernel id * 4 + payload type
std::atomic<int> g_smem_optin[kMaxDevices][kMaxSlots];

// Opts a kernel in to more than 48 KB of dynamic shared memory (once per
// device and size; the largest size opted in so far is kept).
int set_smem(int id, const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return LLMOE_SUCCESS;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LLMOE_ERR_CUDA;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && (size_t)g_smem_optin[dev][id].load(std::memory_order_relaxed) >= bytes) return LLMOE_SUCCESS;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
    cudaGetLastError();
    return LLMOE_ERR_CUDA;
  }
  if (cached) {
    int cur = g_smem_optin[dev][id].load(std::memory_order_relaxed);
    while (cur < (int)bytes && !g_smem_optin[dev][id].compare_exchange_weak(cur, (int)bytes)) {
    }
  }
  return LLMOE_SUCCESS;
}

enum KernelId {
  kRouteKernel = 0,
  kDispatchKernel = 1,
  kCombineKernel = 2,
  kCombinePutKernel = 3,
  kCombineReduceKernel = 4,
  kUnpackKernel = 5,
  kSignaledKernel = 6,
  kCombineKernel4 = 7,
  kCombineKernel2 = 8,
  kCombineReduceRingKernel = 9,
  kDispatchRowsKernel = 10,
  kNumKernels = 11
};
// (dynamic shared memory bytes << 32 | resident CTAs per SM) of the last query
std::atomic<uint64_t> g_occupancy[kMaxDevices][kMaxSlots];

// Cache slot of a kernel instantiation: kernel id and payload type.
int kslot(KernelId id, int dtype = 0) { return (int)id * 4 + dtype; }
static_assert(kNumKernels * 4 <= kMaxSlots, "a cache slot per kernel and payload type");

// Resident CTAs per SM of a kernel at `threads` threads and `smem` bytes of
// dynamic shared memory, cached per device and kernel for the last size
// asked (a kernel's threads are fixed; its shared memory follows the
// geometry).
int blocks_per_sm(int id, const void* fn, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  const bool cached = dev < kMaxDevices && smem < (1ull << 32);
  if (cached) {
    const uint64_t c = g_occupancy[dev][id].load(std::memory_order_relaxed);
    if ((uint32_t)c > 0 && (c >> 32) == smem) return (int)(uint32_t)c;
  }
  int n = 0;
  if (set_smem(id, fn, smem) != LLMOE_SUCCESS) return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 1;
  }
  if (cached) g_occupancy[dev][id].store(((uint64_t)smem << 32) | (uint32_t)n, std::memory_order_relaxed);
  return n;
}

size_t route_smem_bytes(const Geometry& g) {
  const size_t tbk = (size_t)g.TB * g.K;
  return sizeof(int) * ((size_t)g.E + 2 * tbk + (size_t)(g.E & 1));  // pad: 8-byte arrays follow
}

size_t dispatch_smem_bytes(const Geometry& g, bool rows = false) {
  return (size_t)kDspStages * kDspStageBytes + 2 * kDspStages * sizeof(uint64_t) + route_smem_bytes(g) +
         sizeof(uintptr_t) * (size_t)g.TB * g.K * (rows ? 2 : 1);
}

size_t combine_smem_bytes(const Geometry& g) {
  return route_smem_bytes(g) + (sizeof(void*) + sizeof(float)) * (size_t)g.TB * g.K;
}

// Launches with programmatic stream serialization (see wait_prior_grid).
template <typename... KArgs, typename... Args>
int launch(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, llmoe_stream_t stream,
           Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
    cudaGetLastError();  // clear the launch error so it does not leak into later calls
    return LLMOE_ERR_CUDA;
  }
  return LLMOE_SUCCESS;
}

// Workspace of llmoe_dispatch_signaled_static: the per-source completion
// counters live in this fixed device array instead of memory the caller
// allocates.  Every GPU that loads the library holds it until the process
// exits; every call on a device shares it.
constexpr int kStaticMaxRanks = LLMOE_STATIC_MAX_RANKS;
static __device__ __align__(256) int32_t g_static_counters[kStaticMaxRanks + 1];  // per source, plus the consumers'

// The array's device address, looked up once per device (with that device
// current): host code must not hand the symbol itself to a kernel.  The
// address is kept for the life of the process; after a cudaDeviceReset the
// module may be loaded again elsewhere, so the library must not be called on
// a device after it has been reset.
std::atomic<int32_t*> g_static_counters_addr[kMaxDevices];

int static_counters(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return LLMOE_ERR_CUDA;
  }
  if (dev < kMaxDevices) {
    int32_t* c = g_static_counters_addr[dev].load(std::memory_order_acquire);
    if (c != nullptr) {
      *out = c;
      return LLMOE_SUCCESS;
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_counters) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return LLMOE_ERR_CUDA;
  }
  if (dev < kMaxDevices) g_static_counters_addr[dev].store(static_cast<int32_t*>(p), std::memory_order_release);
  *out = static_cast<int32_t*>(p);
  return LLMOE_SUCCESS;
}

// Dispatch and combine grids: R count CTAs, then R * nblk data CTAs (none
// when the call has no tokens).
unsigned count_and_data_ctas(const Geometry& g) {
  return (unsigned)(g.R + (g.T > 0 ? g.R * g.nblk * g.dsplit * g.csplit : 0));
}

// The dispatch launch, with (kRows) or without the experts' input rows.
template <bool kRows>
int launch_dispatch(Geometry& g, const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src,
                    llmoe_stream_t stream) {
  const void* fn = (const void*)dispatch_kernel<kRows>;
  const int id = kslot(kRows ? kDispatchRowsKernel : kDispatchKernel);
  set_blocking(&g, blocks_per_sm(id, fn, kDspThreads, dispatch_smem_bytes(g, kRows)), g.R);
  const int nch_row = (g.row_bytes + kDspChunk - 1) / kDspChunk;
  g.dsplit = g.TB > 1 ? std::max(1, std::min(LLMOE_DSP_SPLIT, nch_row)) : 1;
  const size_t smem = dispatch_smem_bytes(g, kRows);
  int rc = set_smem(id, fn, smem);
  if (rc != LLMOE_SUCCESS) return rc;
  return launch(dispatch_kernel<kRows>, count_and_data_ctas(g), kDspThreads, smem, stream, g, x, topk_idx, recv_x,
                recv_src);
}

template <int DT, int KB>
int launch_combine_kb(Geometry& g, const void* y, const int64_t* topk_idx, const float* topk_w, void* out,
                      llmoe_stream_t stream) {
  const int id = kslot(KB == kKBatch ? kCombineKernel : KB == 4 ? kCombineKernel4 : kCombineKernel2, DT);
  const void* fn = (const void*)combine_kernel<DT, KB>;
  set_blocking(&g, blocks_per_sm(id, fn, kCmbThreads, combine_smem_bytes(g)), g.R);
  // only for blocks of at least 4 tokens: with 2 (a grid of about two
  // waves' tokens) the split leaves a part wave that costs more than it
  // balances (dense16 combine 43.8 -> 46.1 us)
  g.csplit = g.TB >= 4 ? std::max(1, std::min(LLMOE_CMB_SPLIT, g.nchunks)) : 1;
  {
    // the prefetch before the wait (LLMOE_FLAG_INPUTS_READY): about
    // LLMOE_CMB_PREFETCH_BYTES of expert rows over the CTAs of the first wave,
    // at least one unit per warp and at most four.  Measured on DS-V3 (16.8 MB
    // per unit per warp over the grid): one unit saves 1.3 us a round, two 0.8,
    // seven lose 2.7; many-small (4.2 MB per unit) gains from both its units.
    const int64_t resident = std::min<int64_t>((int64_t)g.R * g.nblk * g.csplit, (int64_t)num_sms() * 8);
    const int64_t per_unit = resident * kCmbWarps * g.K * 512;
    g.pf_units = (int)std::max<int64_t>(1, std::min<int64_t>(4, LLMOE_CMB_PREFETCH_BYTES / std::max<int64_t>(per_unit, 1)));
  }
  const size_t smem = combine_smem_bytes(g);
  const int rc = set_smem(id, fn, smem);
  if (rc != LLMOE_SUCCESS) return rc;
  return launch(combine_kernel<DT, KB>, count_and_data_ctas(g), kCmbThreads, smem, stream, g, y, topk_idx, topk_w,
                out);
}

// The kernel whose unrolled load batch is the smallest that holds the
// top-k (2, 4 or 8): with a small top-k the batch of 8 only adds code, and the
// first pass through it, from cold instruction caches, costs time.
template <int DT>
int launch_combine(Geometry& g, const void* y, const int64_t* topk_idx, const float* topk_w, void* out,
                   llmoe_stream_t stream) {
  if (g.K <= 2) return launch_combine_kb<DT, 2>(g, y, topk_idx, topk_w, out, stream);
  if (g.K <= 4) return launch_combine_kb<DT, 4>(g, y, topk_idx, topk_w, out, stream);
  return launch_combine_kb<DT, kKBatch>(g, y, topk_idx, topk_w, out, stream);
}

template <int DT>
int launch_reduce(const Geometry& g, const int64_t* topk_idx, const float* topk_w, void* out, llmoe_stream_t stream) {
  // the ring kernel when a full wave of it has more than one unit per consumer
  // warp (skewed: 1.6, staged combine 37.2 -> 35.3 us; many-small: 0.64, where
  // it took 16.3 us against 14.4)
  const int64_t ring_units = (int64_t)g.R * g.T * ((g.nchunks + kRedWidth - 1) / kRedWidth);
  const size_t smem = reduce_smem_bytes(g);
  int rc = set_smem(kslot(kCombineReduceRingKernel, DT), (const void*)combine_reduce_ring_kernel<DT>, smem);
  if (rc != LLMOE_SUCCESS) return rc;
  const int64_t ring_wave = (int64_t)num_sms() * blocks_per_sm(kslot(kCombineReduceRingKernel, DT),
                                                               (const void*)combine_reduce_ring_kernel<DT>,
                                                               kRedThreads, smem);
  if (ring_units > ring_wave * kRedConsumers) {
    // one wave, each CTA a contiguous range of units
    return launch(combine_reduce_ring_kernel<DT>, (unsigned)ring_wave, kRedThreads, smem, stream, g, topk_idx, topk_w,
                  out);
  }
  const int64_t units = (int64_t)g.R * g.T * g.nchunks;
  const int64_t wave = (int64_t)num_sms() * blocks_per_sm(kslot(kCombineReduceKernel, DT),
                                                          (const void*)combine_reduce_kernel<DT>, kThreads, 0);
  const int64_t blocks = std::min<int64_t>(wave, (units + kThreads / 32 - 1) / (kThreads / 32));
  return launch(combine_reduce_kernel<DT>, (unsigned)blocks, kThreads, 0, stream, g, topk_idx, topk_w, out);
}

#if LLMOE_PHASE_TRACE
// Reference kernels of the trace build, launched the way the data kernels
// are: an empty one, and one whose single thread per CTA loads one cold word,
// to time a launch and a cold load on their own.
__global__ void trace_empty_kernel() {
  release_next_grid();
  wait_prior_grid();
  TRACE(0, threadIdx.x == 0);
}
__global__ void trace_load_kernel(const int64_t* p, int64_t* out) {
  release_next_grid();
  wait_prior_grid();
  TRACE(0, threadIdx.x == 0);
  if (threadIdx.x == 0) {
    const int64_t v = p[blockIdx.x * 4096];
    TRACE(1, true);
    out[blockIdx.x] = v;
  }
}
#endif

// A checked signalled-dispatch launch: geometry, grid and shared memory.
struct SignaledLaunch {
  Geometry g;
  int64_t grid;
  size_t smem;
};

// Every argument and residency check of llmoe_dispatch_signaled (and of its
// static variant) except the workspace pointer; nothing is queued.
int prepare_signaled(const void* x, const int64_t* topk_idx, const void* recv_x, const int32_t* recv_src,
                     int64_t spin_limit, const llmoe_buf_set_t* bs, SignaledLaunch* out) {
  Geometry& g = out->g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if ((g.T > 0 && (x == nullptr || topk_idx == nullptr || !aligned(x, 16) || !aligned(topk_idx, 8))) ||
      recv_x == nullptr || recv_src == nullptr || !aligned(recv_x, 16) || !aligned(recv_src, 4) || spin_limit < 1)
    return LLMOE_ERR_INVALID_ARGUMENT;
  const size_t smem_one = route_smem_bytes(g) + sizeof(uintptr_t) * (size_t)g.K;
  const int occ = blocks_per_sm(kslot(kSignaledKernel), (const void*)dispatch_signaled_kernel, kThreads, smem_one);
  set_blocking(&g, occ);
  out->smem = route_smem_bytes(g) + sizeof(uintptr_t) * (size_t)g.TB * g.K;
  if ((rc = set_smem(kslot(kSignaledKernel), (const void*)dispatch_signaled_kernel, out->smem)) != LLMOE_SUCCESS)
    return rc;
  int fit = 0;  // the exact smem of this launch may lower the occupancy
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, (const void*)dispatch_signaled_kernel, kThreads,
                                                    out->smem) != cudaSuccess) {
    cudaGetLastError();
    return LLMOE_ERR_CUDA;
  }
  out->grid = (int64_t)g.R * g.nblk;
  if (out->grid > (int64_t)num_sms() * fit) return LLMOE_ERR_INVALID_ARGUMENT;  // not all CTAs could be resident
  return LLMOE_SUCCESS;
}

int launch_signaled(const SignaledLaunch& sl, const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src,
                    int32_t* counters, int64_t spin_limit, llmoe_stream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sl.smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, dispatch_signaled_kernel, sl.g, x, topk_idx, recv_x, recv_src, counters,
                         (long long)spin_limit) != cudaSuccess) {
    cudaGetLastError();
    return LLMOE_ERR_CUDA;
  }
  return LLMOE_SUCCESS;
}

}  // namespace

extern "C" {

size_t llmoe_layout_bytes_dtype(int num_max_tokens, int hidden, int num_ranks, int num_experts, int dtype) {
  LayoutInfo li;
  const int es = dtype_size(dtype);
  return es && layout_info(num_max_tokens, hidden, num_ranks, num_experts, es, &li) ? (size_t)li.total : 0;
}

size_t llmoe_layout_bytes(int num_max_tokens, int hidden, int num_ranks, int num_experts) {
  return llmoe_layout_bytes_dtype(num_max_tokens, hidden, num_ranks, num_experts, LLMOE_DTYPE_BF16);
}

int llmoe_layout_offsets(int num_max_tokens, int hidden, int num_ranks, int num_experts, int set,
                         uint64_t* send_offset, uint64_t* recv_offset, uint64_t* signal_offset) {
  return llmoe_layout_offsets_dtype(num_max_tokens, hidden, num_ranks, num_experts, LLMOE_DTYPE_BF16, set,
                                    send_offset, recv_offset, signal_offset);
}

int llmoe_layout_offsets_dtype(int num_max_tokens, int hidden, int num_ranks, int num_experts, int dtype, int set,
                               uint64_t* send_offset, uint64_t* recv_offset, uint64_t* signal_offset) {
  LayoutInfo li;
  const int es = dtype_size(dtype);
  if ((set != 0 && set != 1) || es == 0 || !layout_info(num_max_tokens, hidden, num_ranks, num_experts, es, &li))
    return LLMOE_ERR_INVALID_ARGUMENT;
  if (send_offset) *send_offset = li.send * (uint64_t)set;
  if (recv_offset) *recv_offset = 2 * li.send + li.recv * (uint64_t)set;
  if (signal_offset) *signal_offset = 2 * li.send + 2 * li.recv + li.sig * (uint64_t)set;
  return LLMOE_SUCCESS;
}

int llmoe_route(const int64_t* topk_idx, int32_t* slot, int64_t* counts, const llmoe_buf_set_t* bs,
                llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, false, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (counts == nullptr || !aligned(counts, 8)) return LLMOE_ERR_INVALID_ARGUMENT;
  if (g.T > 0 && (topk_idx == nullptr || slot == nullptr || !aligned(topk_idx, 8) || !aligned(slot, 4)))
    return LLMOE_ERR_INVALID_ARGUMENT;
  set_blocking(&g, blocks_per_sm(kslot(kRouteKernel), (const void*)route_kernel, kThreads, route_smem_bytes(g)));
  const size_t smem = route_smem_bytes(g);
  if ((rc = set_smem(kslot(kRouteKernel), (const void*)route_kernel, smem)) != LLMOE_SUCCESS) return rc;
  return launch(route_kernel, g.R * g.nblk, kThreads, smem, stream, g, topk_idx, slot, counts);
}

int llmoe_dispatch(const void* x, const int64_t* topk_idx, const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (g.T > 0 && (x == nullptr || topk_idx == nullptr || !aligned(x, 16) || !aligned(topk_idx, 8)))
    return LLMOE_ERR_INVALID_ARGUMENT;
  return launch_dispatch<false>(g, x, topk_idx, nullptr, nullptr, stream);
}

int llmoe_dispatch_unpack(const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src,
                          const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (g.T > 0 && (x == nullptr || topk_idx == nullptr || !aligned(x, 16) || !aligned(topk_idx, 8)))
    return LLMOE_ERR_INVALID_ARGUMENT;
  if (recv_x == nullptr || recv_src == nullptr || !aligned(recv_x, 16) || !aligned(recv_src, 4))
    return LLMOE_ERR_INVALID_ARGUMENT;
  return launch_dispatch<true>(g, x, topk_idx, recv_x, recv_src, stream);
}

int llmoe_combine(const void* y, const int64_t* topk_idx, const float* topk_w, void* out,
                  const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (g.T > 0 && (y == nullptr || topk_idx == nullptr || topk_w == nullptr || out == nullptr || !aligned(y, 16) ||
                  !aligned(out, 16) || !aligned(topk_idx, 8) || !aligned(topk_w, 4)))
    return LLMOE_ERR_INVALID_ARGUMENT;
  if (g.T > 0) {
    // out must not overlap y
    const uintptr_t yb = reinterpret_cast<uintptr_t>(y), ob = reinterpret_cast<uintptr_t>(out);
    const uintptr_t ye = yb + (uintptr_t)g.E * g.R * g.T_max * g.row_bytes, oe = ob + (uintptr_t)g.R * g.T * g.row_bytes;
    if (ob < ye && yb < oe) return LLMOE_ERR_INVALID_ARGUMENT;
  }
  switch (g.dtype) {
    case LLMOE_DTYPE_FP16: return launch_combine<LLMOE_DTYPE_FP16>(g, y, topk_idx, topk_w, out, stream);
    case LLMOE_DTYPE_FP32: return launch_combine<LLMOE_DTYPE_FP32>(g, y, topk_idx, topk_w, out, stream);
    default: return launch_combine<LLMOE_DTYPE_BF16>(g, y, topk_idx, topk_w, out, stream);
  }
}

int llmoe_combine_staged(const void* y, const int64_t* topk_idx, const float* topk_w, void* out,
                         const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (g.T > 0 && (y == nullptr || topk_idx == nullptr || topk_w == nullptr || out == nullptr || !aligned(y, 16) ||
                  !aligned(out, 16) || !aligned(topk_idx, 8) || !aligned(topk_w, 4)))
    return LLMOE_ERR_INVALID_ARGUMENT;
  if (g.T > 0) {
    const uintptr_t yb = reinterpret_cast<uintptr_t>(y), ob = reinterpret_cast<uintptr_t>(out);
    const uintptr_t ye = yb + (uintptr_t)g.E * g.R * g.T_max * g.row_bytes, oe = ob + (uintptr_t)g.R * g.T * g.row_bytes;
    if (ob < ye && yb < oe) return LLMOE_ERR_INVALID_ARGUMENT;
  }
  const size_t put_extra = (sizeof(void*) + sizeof(uintptr_t)) * (size_t)g.K;
  set_blocking(&g, LLMOE_PUT_WAVES * blocks_per_sm(kslot(kCombinePutKernel), (const void*)combine_put_kernel, kThreads,
                                 route_smem_bytes(g) + put_extra));
  const size_t smem = route_smem_bytes(g) + (sizeof(void*) + sizeof(uintptr_t)) * (size_t)g.TB * g.K;
  if ((rc = set_smem(kslot(kCombinePutKernel), (const void*)combine_put_kernel, smem)) != LLMOE_SUCCESS) return rc;
  if ((rc = launch(combine_put_kernel, g.R * g.nblk, kThreads, smem, stream, g, y, topk_idx)) != LLMOE_SUCCESS)
    return rc;
  if (g.T == 0) return LLMOE_SUCCESS;
  Geometry gr = g;
  gr.flags &= ~LLMOE_FLAG_CLEAN_OTHER_SET;  // the put kernel already cleaned
  switch (g.dtype) {
    case LLMOE_DTYPE_FP16: return launch_reduce<LLMOE_DTYPE_FP16>(gr, topk_idx, topk_w, out, stream);
    case LLMOE_DTYPE_FP32: return launch_reduce<LLMOE_DTYPE_FP32>(gr, topk_idx, topk_w, out, stream);
    default: return launch_reduce<LLMOE_DTYPE_BF16>(gr, topk_idx, topk_w, out, stream);
  }
}

int llmoe_unpack(void* recv_x, int32_t* recv_src, const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (recv_x == nullptr || recv_src == nullptr || !aligned(recv_x, 16) || !aligned(recv_src, 4))
    return LLMOE_ERR_INVALID_ARGUMENT;
  // the balanced kernel pays for a scan of every bucket count in every CTA;
  // with at least as many buckets as routed entries there is little skew to
  // balance and the per-bucket kernel is cheaper
  const int64_t nb = (int64_t)g.E * g.R, entries = (int64_t)g.R * g.T * g.K;
  if (nb <= kMaxScanBuckets && nb < entries) {
    // one full wave: the copy is latency-bound, so every resident warp helps
    const int64_t wave = (int64_t)num_sms() * blocks_per_sm(kslot(kUnpackKernel, 1),
                                                            (const void*)unpack_balanced_kernel, kUnpackThreads, 0);
    return launch(unpack_balanced_kernel, (unsigned)wave, kUnpackThreads, 0, stream, g, recv_x, recv_src);
  }
  const int64_t wave =
      (int64_t)num_sms() * blocks_per_sm(kslot(kUnpackKernel), (const void*)unpack_kernel, kThreads, 0);
  const int64_t blocks = std::min<int64_t>(wave, ((int64_t)g.E * g.R + kThreads / 32 - 1) / (kThreads / 32));
  return launch(unpack_kernel, (unsigned)blocks, kThreads, 0, stream, g, recv_x, recv_src);
}

size_t llmoe_signal_workspace_bytes(const llmoe_buf_set_t* bs) {
  if (bs == nullptr || bs->num_ranks < 1) return 0;
  return ((size_t)(bs->num_ranks + 1) * sizeof(int32_t) + 255) / 256 * 256;  // per source, plus the consumers'
}

int llmoe_dispatch_signaled(const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src, void* workspace,
                            int64_t spin_limit, const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  SignaledLaunch sl;
  const int rc = prepare_signaled(x, topk_idx, recv_x, recv_src, spin_limit, bs, &sl);
  if (rc != LLMOE_SUCCESS) return rc;
  if (workspace == nullptr || !aligned(workspace, 4)) return LLMOE_ERR_INVALID_ARGUMENT;
  return launch_signaled(sl, x, topk_idx, recv_x, recv_src, static_cast<int32_t*>(workspace), spin_limit, stream);
}

int llmoe_dispatch_signaled_static(const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src,
                                   int64_t spin_limit, const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  if (bs == nullptr || bs->num_ranks < 1) return LLMOE_ERR_INVALID_ARGUMENT;
  if (bs->num_ranks > kStaticMaxRanks) return LLMOE_ERR_INVALID_ARGUMENT;  // more ranks than the array holds
  // every check before anything is queued: a rejected call leaves the
  // shared counters alone
  SignaledLaunch sl;
  int rc = prepare_signaled(x, topk_idx, recv_x, recv_src, spin_limit, bs, &sl);
  if (rc != LLMOE_SUCCESS) return rc;
  int32_t* counters = nullptr;
  if ((rc = static_counters(&counters)) != LLMOE_SUCCESS) return rc;
  // the counters must start at zero; clear the part this call uses, in
  // stream order
  if (cudaMemsetAsync(counters, 0, sizeof(int32_t) * (size_t)(bs->num_ranks + 1), (cudaStream_t)stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return LLMOE_ERR_CUDA;
  }
  return launch_signaled(sl, x, topk_idx, recv_x, recv_src, counters, spin_limit, stream);
}

int llmoe_clean(const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  const int64_t n = (int64_t)g.R * g.E;
  int blocks = (int)((n + kThreads - 1) / kThreads);
  if (blocks > 64) blocks = 64;
  return launch(clean_kernel, blocks, kThreads, 0, stream, g.base, g.rank_stride, g.sig_off, g.R, g.E);
}

int llmoe_get_error(const llmoe_buf_set_t* bs, llmoe_stream_t stream, int32_t* code, int reset) {
  if (bs == nullptr || code == nullptr) return LLMOE_ERR_INVALID_ARGUMENT;
  if (bs->err == nullptr) return LLMOE_ERR_INVALID_USAGE;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, bs->err, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return LLMOE_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LLMOE_ERR_CUDA;
  if (reset) {
    if (cudaMemsetAsync(bs->err, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess) return LLMOE_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LLMOE_ERR_CUDA;
  }
  *code = v;
  return LLMOE_SUCCESS;
}

#if LLMOE_PHASE_TRACE
// Trace build only (not declared in llmoe.h): copy the per-CTA stamps of the
// last traced launches out, clear them, and time the two reference kernels.
LLMOE_API int llmoe_phase_trace_read(unsigned long long* host, int max_ctas) {
  const int n = std::min(max_ctas, kTraceCtas);
  if (host == nullptr || n < 1) return LLMOE_ERR_INVALID_ARGUMENT;
  if (cudaMemcpyFromSymbol(host, g_phase_trace, sizeof(unsigned long long) * 2 * kTracePhases * (size_t)n) !=
      cudaSuccess)
    return LLMOE_ERR_CUDA;
  return LLMOE_SUCCESS;
}
LLMOE_API int llmoe_phase_trace_clear(llmoe_stream_t stream) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_phase_trace) != cudaSuccess) return LLMOE_ERR_CUDA;
  return cudaMemsetAsync(p, 0, sizeof(g_phase_trace), (cudaStream_t)stream) == cudaSuccess ? LLMOE_SUCCESS
                                                                                            : LLMOE_ERR_CUDA;
}
LLMOE_API int llmoe_trace_empty(int ctas, llmoe_stream_t stream) {
  return launch(trace_empty_kernel, (unsigned)ctas, kThreads, 0, stream);
}
// p: ctas * 4096 int64 words (one cold word 32 KB apart per CTA), out: ctas words
LLMOE_API int llmoe_trace_load(const int64_t* p, int64_t* out, int ctas, llmoe_stream_t stream) {
  return launch(trace_load_kernel, (unsigned)ctas, kThreads, 0, stream, p, out);
}
#endif

const char* llmoe_status_string(int status) {
  switch (status) {
    case LLMOE_SUCCESS: return "success";
    case LLMOE_ERR_CUDA: return "CUDA error";
    case LLMOE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case LLMOE_ERR_INVALID_USAGE: return "invalid usage";
    default: return "unknown status";
  }
}

}  // extern "C"
