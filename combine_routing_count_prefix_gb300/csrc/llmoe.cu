// llmoe.cu -- sm_103a kernels and the C ABI of libllmoe.so (see include/llmoe.h).
//
// One GPU holds R simulated expert-parallel ranks as R segments of one
// allocation, each laid out as LLMoEBufferLayout<bf16> (LL_MoE_Buffers.hpp).
// The data path is pure movement plus one fp32 multiply-add per byte pair, so
// it is bound by HBM bandwidth: no tensor cores, 16-byte vector accesses,
// every row read once.
//
// Kernels:
//   route_scan (device function, run at the start of the route, dispatch and
//     combine kernels): per-(expert, source rank) counts and slots, where the
//     slot of token t for expert e is the number of earlier tokens of the same
//     source rank that chose e.  Built from a shared-memory histogram of the
//     tokens before the CTA's block (integer atomics, so the result does not
//     depend on their order) plus an in-block rank.  No global atomics, no
//     scratch memory.
//   dispatch_kernel: each warp moves 32 quads (512 B) of one token row per
//     unit and writes them to the K destination messages.  A message is
//     4 + 2H bytes, which is 4 (mod 16) for H % 8 == 0, so a destination row
//     starts at any 4-byte phase; the warp shifts its quads by whole 32-bit
//     words (neighbour quad via a shuffle) and issues aligned 16-byte stores,
//     with 4/8-byte stores only at the head and tail of each message.
//   combine_kernel: each warp reduces 32 quads of one output row: K aligned
//     16-byte loads of expert rows, fp32 products rounded then added in
//     ascending k (__fmul_rn / __fadd_rn: never contracted to an FMA), bf16
//     round-to-nearest-even store.
//   clean_kernel: zeroes a set's R * E signal words (LLMoEBuffer::clean_meta).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include "llmoe.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTokensPerBlock = 32;
constexpr int kKBatch = 8;  // expert rows loaded before accumulating, combine

struct Geometry {
  uint8_t* base;         // rank 0's buffer
  uint64_t rank_stride;  // bytes between rank buffers
  uint64_t recv_off;     // this set's receive region, from a rank buffer's start
  uint64_t sig_off;      // this set's signal words
  uint64_t msg;          // 4 + 2H
  int32_t* err;          // optional error word
  int T_max, T, H, R, E, K, L;
  int nq;       // 16-byte quads per row, H / 8
  int nchunks;  // warp units per row, ceil(nq / 32)
  int TB;       // tokens per CTA
  int nblk;     // token blocks per source rank
};

__device__ __forceinline__ void report(int32_t* err, int32_t code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// Shared-memory view used by the three route-scan kernels.
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

// Routing count / prefix scan for tokens [t0, t1) of source rank src.
// On return (after a __syncthreads): s.slot[q] for q = (t - t0) * K + k, and,
// when full_counts, s.hist[e] = number of entries of src choosing e over all
// of the call's tokens.
__device__ void route_scan(const Geometry& g, const int64_t* __restrict__ idx, int src, int t0, int t1,
                           bool full_counts, const RouteSmem& s) {
  const int tid = threadIdx.x;
  const int K = g.K, E = g.E;
  for (int e = tid; e < E; e += blockDim.x) s.hist[e] = 0;
  const int64_t* src_idx = idx + (int64_t)src * g.T * K;
  const int nblock = (t1 - t0) * K;
  for (int q = tid; q < nblock; q += blockDim.x) {
    int64_t e = src_idx[(int64_t)t0 * K + q];
    s.ent[q] = (e >= 0 && e < E) ? (int)e : -1;
    if (e < -1 || e >= E) report(g.err, LLMOE_DEV_BAD_EXPERT);
  }
  __syncthreads();
  // histogram of the tokens before the block
  const int npre = t0 * K;
  for (int i = tid; i < npre; i += blockDim.x) {
    int64_t e = src_idx[i];
    if (e >= 0 && e < E) atomicAdd(&s.hist[e], 1);
  }
  __syncthreads();
  // slot = earlier tokens before the block + earlier tokens inside it
  for (int q = tid; q < nblock; q += blockDim.x) {
    const int e = s.ent[q];
    int sl = -1;
    if (e >= 0) {
      const int tl = q / K, k = q % K;
      int r = 0;
      for (int p = 0; p < tl * K; ++p) r += (s.ent[p] == e);
      for (int k2 = 0; k2 < k; ++k2)
        if (s.ent[tl * K + k2] == e) report(g.err, LLMOE_DEV_DUPLICATE);
      sl = s.hist[e] + r;
      if (sl >= g.T_max) {  // only reachable when a token repeats an expert
        report(g.err, LLMOE_DEV_SLOT_RANGE);
        sl = -1;
      }
    }
    s.slot[q] = sl;
  }
  __syncthreads();
  if (full_counts) {
    for (int q = tid; q < nblock; q += blockDim.x)
      if (s.ent[q] >= 0) atomicAdd(&s.hist[s.ent[q]], 1);
    __syncthreads();
  }
}

// Writes rank dst's (dispatch) or rank src's (combine) signal words from the
// full histogram; checks that each word was zero (cleaned) in validate mode.
__device__ __forceinline__ void put_signal(const Geometry& g, int64_t* word, int value) {
  if (g.err != nullptr && *reinterpret_cast<volatile int64_t*>(word) != 0) report(g.err, LLMOE_DEV_STALE_SIGNAL);
  *word = (int64_t)value;
}

__device__ __forceinline__ uint4 ldg16(const uint4* p) { return __ldg(p); }

__device__ __forceinline__ uint4 shfl_up16(uint4 v, int lane_delta) {
  uint4 r;
  r.x = __shfl_up_sync(0xffffffffu, v.x, lane_delta);
  r.y = __shfl_up_sync(0xffffffffu, v.y, lane_delta);
  r.z = __shfl_up_sync(0xffffffffu, v.z, lane_delta);
  r.w = __shfl_up_sync(0xffffffffu, v.w, lane_delta);
  return r;
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

__device__ __forceinline__ void st16(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void st8(uint8_t* p, uint32_t a, uint32_t b) {
  *reinterpret_cast<uint2*>(p) = make_uint2(a, b);
}
__device__ __forceinline__ void st4(uint8_t* p, uint32_t a) { *reinterpret_cast<uint32_t*>(p) = a; }

// Writes source quad j of a token row (and the header / tail pieces that fall
// to it) into the message at `msg_addr`.  prev is quad j-1, or (0,0,0,t) for
// j == 0 so that prev.w is the header.
__device__ __forceinline__ void put_quad(uint8_t* msg_addr, int j, int nq, const uint4& prev, const uint4& cur) {
  uint8_t* pa = msg_addr + 4;  // payload
  const int phase = (int)((reinterpret_cast<uintptr_t>(pa) >> 2) & 3);
  uint8_t* qb = pa - 4 * phase;  // 16-byte aligned
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

__global__ void __launch_bounds__(kThreads) dispatch_kernel(Geometry g, const uint16_t* __restrict__ x,
                                                            const int64_t* __restrict__ idx) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  uint8_t** s_dst = reinterpret_cast<uint8_t**>(s.slot + g.TB * g.K + (g.E & 1));

  const int src = blockIdx.x / g.nblk, b = blockIdx.x % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const bool last = (b == g.nblk - 1);
  route_scan(g, idx, src, t0, t1, last, s);

  const int nblock = (t1 - t0) * g.K;
  for (int q = threadIdx.x; q < nblock; q += blockDim.x) {
    const int e = s.ent[q], sl = s.slot[q];
    uint8_t* d = nullptr;
    if (e >= 0 && sl >= 0) {
      const int dst = e / g.L, le = e % g.L;
      const uint64_t row = ((uint64_t)le * g.R + src) * g.T_max + sl;
      d = g.base + dst * g.rank_stride + g.recv_off + row * g.msg;
    }
    s_dst[q] = d;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nunits = (t1 - t0) * g.nchunks;
  for (int u = warp; u < nunits; u += kWarps) {
    const int tl = u / g.nchunks, c = u % g.nchunks;
    const int t = t0 + tl;
    const uint4* xrow = reinterpret_cast<const uint4*>(x + ((int64_t)src * g.T + t) * g.H);
    const int j = c * 32 + lane;
    uint4 cur = make_uint4(0, 0, 0, 0);
    if (j < g.nq) cur = ldg16(xrow + j);
    uint4 prev = shfl_up16(cur, 1);
    if (lane == 0) prev = (j == 0) ? make_uint4(0, 0, 0, (uint32_t)t) : ldg16(xrow + j - 1);
    if (j < g.nq) {
      uint8_t* const* dsts = s_dst + tl * g.K;
      for (int k = 0; k < g.K; ++k) {
        uint8_t* d = dsts[k];
        if (d != nullptr) put_quad(d, j, g.nq, prev, cur);
      }
    }
  }

  if (last) {
    // rank dst's word le * R + src = count of bucket (le, src)
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      const int dst = e / g.L, le = e % g.L;
      int64_t* w = reinterpret_cast<int64_t*>(g.base + dst * g.rank_stride + g.sig_off) + ((int64_t)le * g.R + src);
      put_signal(g, w, s.hist[e]);
    }
  }
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void axpy_quad(float (&acc)[8], float w, const uint4& v) {
  acc[0] = __fadd_rn(acc[0], __fmul_rn(w, bf16lo(v.x)));
  acc[1] = __fadd_rn(acc[1], __fmul_rn(w, bf16hi(v.x)));
  acc[2] = __fadd_rn(acc[2], __fmul_rn(w, bf16lo(v.y)));
  acc[3] = __fadd_rn(acc[3], __fmul_rn(w, bf16hi(v.y)));
  acc[4] = __fadd_rn(acc[4], __fmul_rn(w, bf16lo(v.z)));
  acc[5] = __fadd_rn(acc[5], __fmul_rn(w, bf16hi(v.z)));
  acc[6] = __fadd_rn(acc[6], __fmul_rn(w, bf16lo(v.w)));
  acc[7] = __fadd_rn(acc[7], __fmul_rn(w, bf16hi(v.w)));
}

__global__ void __launch_bounds__(kThreads) combine_kernel(Geometry g, const uint16_t* __restrict__ y,
                                                           const int64_t* __restrict__ idx,
                                                           const float* __restrict__ topk_w,
                                                           uint16_t* __restrict__ out) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  const int TBK = g.TB * g.K;
  const uint4** s_row = reinterpret_cast<const uint4**>(s.slot + TBK + (g.E & 1));
  float* s_w = reinterpret_cast<float*>(s_row + TBK);

  const int src = blockIdx.x / g.nblk, b = blockIdx.x % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const bool last = (b == g.nblk - 1);
  route_scan(g, idx, src, t0, t1, last, s);

  const int nblock = (t1 - t0) * g.K;
  for (int q = threadIdx.x; q < nblock; q += blockDim.x) {
    const int e = s.ent[q], sl = s.slot[q];
    const uint4* r = nullptr;
    if (e >= 0 && sl >= 0) {
      const uint64_t row = (uint64_t)e * g.R * g.T_max + (uint64_t)src * g.T_max + sl;
      r = reinterpret_cast<const uint4*>(y + row * g.H);
    }
    s_row[q] = r;
    s_w[q] = topk_w[((int64_t)src * g.T + t0) * g.K + q];
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nunits = (t1 - t0) * g.nchunks;
  for (int u = warp; u < nunits; u += kWarps) {
    const int tl = u / g.nchunks, c = u % g.nchunks;
    const int t = t0 + tl;
    const int j = c * 32 + lane;
    if (j >= g.nq) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const uint4* const* rows = s_row + tl * g.K;
    const float* ws = s_w + tl * g.K;
    for (int k0 = 0; k0 < g.K; k0 += kKBatch) {
      uint4 v[kKBatch];
#pragma unroll
      for (int i = 0; i < kKBatch; ++i) {
        const int k = k0 + i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (k < g.K && rows[k] != nullptr) v[i] = ldg16(rows[k] + j);
      }
#pragma unroll
      for (int i = 0; i < kKBatch; ++i) {
        const int k = k0 + i;
        if (k < g.K && rows[k] != nullptr) axpy_quad(acc, ws[k], v[i]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + ((int64_t)src * g.T + t) * g.H)[j] = o;
  }

  if (last) {
    // rank src's word e = rows expert e returns to src
    int64_t* w = reinterpret_cast<int64_t*>(g.base + src * g.rank_stride + g.sig_off);
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) put_signal(g, w + e, s.hist[e]);
  }
}

__global__ void __launch_bounds__(kThreads) route_kernel(Geometry g, const int64_t* __restrict__ idx,
                                                         int32_t* __restrict__ slot_out,
                                                         int64_t* __restrict__ counts) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RouteSmem s = carve_route(smem, g);
  const int src = blockIdx.x / g.nblk, b = blockIdx.x % g.nblk;
  const int t0 = b * g.TB, t1 = min(g.T, t0 + g.TB);
  const bool last = (b == g.nblk - 1);
  route_scan(g, idx, src, t0, t1, last, s);
  const int nblock = (t1 - t0) * g.K;
  for (int q = threadIdx.x; q < nblock; q += blockDim.x)
    slot_out[((int64_t)src * g.T + t0) * g.K + q] = s.slot[q];
  if (last)
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) counts[(int64_t)e * g.R + src] = s.hist[e];
}

__global__ void __launch_bounds__(kThreads) clean_kernel(uint8_t* base, uint64_t rank_stride, uint64_t sig_off,
                                                         int R, int E) {
  const int64_t n = (int64_t)R * E;
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

// LLMoEBufferLayout<bf16>: send = max(T*msg, E*T*msg), recv = E*T*msg (both
// roles), sig = 8*E; each region twice; msg = sizeof(int) + 2*hidden.
bool layout_info(int T, int H, int R, int E, LayoutInfo* out) {
  if (T < 1 || H < 1 || R < 1 || E < 1) return false;
  uint64_t msg, et, dsend, csend, recv, total = 0, two;
  if (!mul_u64((uint64_t)H, 2, &msg) || !add_u64(msg, 4, &msg)) return false;
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

int g_num_sms[64] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && g_num_sms[dev] > 0) return g_num_sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) g_num_sms[dev] = n;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validates a buffer set and fills the launch geometry.  need_buffers: the
// call writes the rank buffers (base / rank_stride / set must be valid).
int make_geometry(const llmoe_buf_set_t* bs, bool need_buffers, Geometry* g) {
  if (bs == nullptr) return LLMOE_ERR_INVALID_ARGUMENT;
  const int T_max = bs->num_max_tokens, T = bs->num_tokens, H = bs->hidden, R = bs->num_ranks,
            E = bs->num_experts, K = bs->num_topk;
  if (T_max < 1 || T < 0 || T > T_max || H < 8 || H % 8 != 0 || R < 1 || E < R || E % R != 0 ||
      E > LLMOE_MAX_EXPERTS || K < 1 || K > LLMOE_MAX_TOPK || K > E)
    return LLMOE_ERR_INVALID_ARGUMENT;
  const int set = need_buffers ? bs->set : 0;
  if (set != 0 && set != 1) return LLMOE_ERR_INVALID_ARGUMENT;
  if (bs->err != nullptr && !aligned(bs->err, 4)) return LLMOE_ERR_INVALID_ARGUMENT;
  LayoutInfo li;
  if (!layout_info(T_max, H, R, E, &li)) return LLMOE_ERR_INVALID_ARGUMENT;
  // every index the kernels form stays below 2^63
  uint64_t rows, elems;
  if (!mul_u64((uint64_t)E * (uint64_t)R, (uint64_t)T_max, &rows) || !mul_u64(rows, (uint64_t)H, &elems) ||
      elems > (uint64_t)INT64_MAX / 2)
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
  g->msg = li.msg;
  g->err = bs->err;
  g->T_max = T_max;
  g->T = T;
  g->H = H;
  g->R = R;
  g->E = E;
  g->K = K;
  g->L = E / R;
  g->nq = H / 8;
  g->nchunks = (g->nq + 31) / 32;
  // tokens per CTA: enough CTAs for about 8 resident per SM, at most 32 tokens
  const int64_t tokens = (int64_t)R * T;
  const int64_t target = (int64_t)num_sms() * 8;
  int64_t tb = (tokens + target - 1) / target;
  if (tb < 1) tb = 1;
  if (tb > kMaxTokensPerBlock) tb = kMaxTokensPerBlock;
  g->TB = (int)tb;
  g->nblk = T > 0 ? (T + g->TB - 1) / g->TB : 1;
  return LLMOE_SUCCESS;
}

size_t route_smem_bytes(const Geometry& g) {
  const size_t tbk = (size_t)g.TB * g.K;
  return sizeof(int) * ((size_t)g.E + 2 * tbk + (size_t)(g.E & 1));  // pad: 8-byte arrays follow
}

int set_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return LLMOE_SUCCESS;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return LLMOE_ERR_CUDA;
  return LLMOE_SUCCESS;
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? LLMOE_SUCCESS : LLMOE_ERR_CUDA; }

}  // namespace

extern "C" {

size_t llmoe_layout_bytes(int num_max_tokens, int hidden, int num_ranks, int num_experts) {
  LayoutInfo li;
  return layout_info(num_max_tokens, hidden, num_ranks, num_experts, &li) ? (size_t)li.total : 0;
}

int llmoe_layout_offsets(int num_max_tokens, int hidden, int num_ranks, int num_experts, int set,
                         uint64_t* send_offset, uint64_t* recv_offset, uint64_t* signal_offset) {
  LayoutInfo li;
  if ((set != 0 && set != 1) || !layout_info(num_max_tokens, hidden, num_ranks, num_experts, &li))
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
  const size_t smem = route_smem_bytes(g);
  if ((rc = set_smem((const void*)route_kernel, smem)) != LLMOE_SUCCESS) return rc;
  route_kernel<<<g.R * g.nblk, kThreads, smem, (cudaStream_t)stream>>>(g, topk_idx, slot, counts);
  return launch_status();
}

int llmoe_dispatch(const uint16_t* x, const int64_t* topk_idx, const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  if (g.T > 0 && (x == nullptr || topk_idx == nullptr || !aligned(x, 16) || !aligned(topk_idx, 8)))
    return LLMOE_ERR_INVALID_ARGUMENT;
  const size_t tbk = (size_t)g.TB * g.K;
  const size_t smem = route_smem_bytes(g) + sizeof(void*) * tbk;
  if ((rc = set_smem((const void*)dispatch_kernel, smem)) != LLMOE_SUCCESS) return rc;
  dispatch_kernel<<<g.R * g.nblk, kThreads, smem, (cudaStream_t)stream>>>(g, x, topk_idx);
  return launch_status();
}

int llmoe_combine(const uint16_t* y, const int64_t* topk_idx, const float* topk_w, uint16_t* out,
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
    const uintptr_t ye = yb + (uintptr_t)g.E * g.R * g.T_max * g.H * 2, oe = ob + (uintptr_t)g.R * g.T * g.H * 2;
    if (ob < ye && yb < oe) return LLMOE_ERR_INVALID_ARGUMENT;
  }
  const size_t tbk = (size_t)g.TB * g.K;
  const size_t smem = route_smem_bytes(g) + (sizeof(void*) + sizeof(float)) * tbk;
  if ((rc = set_smem((const void*)combine_kernel, smem)) != LLMOE_SUCCESS) return rc;
  combine_kernel<<<g.R * g.nblk, kThreads, smem, (cudaStream_t)stream>>>(g, y, topk_idx, topk_w, out);
  return launch_status();
}

int llmoe_clean(const llmoe_buf_set_t* bs, llmoe_stream_t stream) {
  Geometry g;
  int rc = make_geometry(bs, true, &g);
  if (rc != LLMOE_SUCCESS) return rc;
  const int64_t n = (int64_t)g.R * g.E;
  int blocks = (int)((n + kThreads - 1) / kThreads);
  if (blocks > 64) blocks = 64;
  clean_kernel<<<blocks, kThreads, 0, (cudaStream_t)stream>>>(g.base, g.rank_stride, g.sig_off, g.R, g.E);
  return launch_status();
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
