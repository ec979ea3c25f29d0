/*
 * llmoe_oracle.c -- plain, slow, single-threaded CPU oracle for the low-latency
 * MoE dispatch / combine data path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this code.  The CUDA library never
 * links it, includes it or calls it, and it shares no source with the CUDA
 * library.
 *
 * What it follows:
 *   - LL_MoE_Buffers.hpp (rocshmem LL_MoE example), struct LLMoEBufferLayout,
 *     constructor: message sizes, send-buffer sizes, receive-buffer sizes,
 *     signaling buffers, pointer assignment for the two buffer sets, and
 *     get_rdma_size_hint (which returns total_bytes).
 *   - LL_MoE_Buffers.hpp, struct LLMoEBuffer: the roles of the dispatch
 *     recv buffer ([num_experts * num_tokens] messages), the recv-count words
 *     ([num_experts] int64), the combine buffers and the recv-flag words, and
 *     clean_meta(): one zeroing of num_sig_elems int64 words resets both the
 *     dispatch counts and the combine flags of a set.
 *   - Where the header leaves a step open (what the int header holds, how the
 *     receive rows are indexed, the order inside a bucket, the meaning of the
 *     signal words, the accumulation order of the combine) this file takes the
 *     readings written next to each function.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared.  -ffp-contract=off
 * matters: the combine's "round the product, then round the sum" must not be
 * fused into an FMA (gcc contracts by default on aarch64).
 *
 * Pin status: every function here is pinned by a CPU test (layout by a closed
 * form and a worked value, the route scan by brute force against a sort-based
 * formulation, dispatch by round trip, combine by closed forms and identity
 * experts, the bf16 rounding by hand-built bit patterns and a library cast).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORACLE_OK 0
#define ORACLE_BAD_EXPERT 1   /* an id outside [-1, num_experts) */
#define ORACLE_DUPLICATE 2    /* the same expert twice in one token */
#define ORACLE_BAD_ARG (-1)   /* a dimension < 1, or num_tokens > num_max_tokens */
#define ORACLE_ASSERT (-2)    /* the layout's "% sizeof(int) == 0" assertion fails */
#define ORACLE_OVERFLOW (-3)  /* a byte count does not fit in 64 bits */

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a binary32 to the nearest bfloat16, ties to the even neighbour
 * (IEEE 754 roundTiesToEven applied to the 16 dropped fraction bits).  A NaN
 * stays a NaN (quiet bit set); the data path never produces one. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t kept = u >> 16;          /* sign, exponent, top 7 fraction bits */
  uint32_t dropped = u & 0xffffu;   /* the part that is rounded away */
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;            /* a carry into the exponent is correct */
}

void oracle_f32_to_bf16_array(const float* f, uint16_t* b, int64_t n) {
  for (int64_t i = 0; i < n; ++i) b[i] = oracle_f32_to_bf16(f[i]);
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Widening to binary32 is exact. */
float oracle_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) << 31;
  uint32_t exp = (h >> 10) & 0x1fu, frac = h & 0x3ffu, u;
  if (exp == 0) {
    /* zero or subnormal: frac * 2^-24, exact in binary32 */
    float mag = (float)frac * 5.9604644775390625e-08f;
    float f = sign ? -mag : mag;
    return f;
  }
  if (exp == 31) {
    u = sign | 0x7f800000u | (frac << 13); /* inf or NaN */
  } else {
    u = sign | ((exp - 15 + 127) << 23) | (frac << 13);
  }
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round half to even of a non-negative value below 2^24 that is an integer
 * plus a fraction representable in binary32 (as every value scaled here is). */
static uint32_t round_half_even_u(float q) {
  float fl = (float)(uint32_t)q; /* truncation = floor for q >= 0 */
  float r = q - fl;              /* exact */
  uint32_t n = (uint32_t)fl;
  if (r > 0.5f || (r == 0.5f && (n & 1u))) n += 1u;
  return n;
}

/* binary32 -> binary16, round to nearest, ties to even; overflow to
 * infinity; NaN stays NaN. */
uint16_t oracle_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);
  float a = fabsf(f);
  if (a >= 65520.0f) return (uint16_t)(sign | 0x7c00u); /* at or past the midpoint above 65504 */
  if (a < 6.103515625e-05f) {                           /* below 2^-14: subnormal step 2^-24 */
    uint32_t n = round_half_even_u(a * 16777216.0f);    /* a / 2^-24, exact scaling */
    return (uint16_t)(sign | n);                        /* n == 1024 is the smallest normal */
  }
  int e;
  float m = frexpf(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
  int exp = e - 1;                       /* a = (2m) * 2^exp, 2m in [1, 2) */
  float q = (2.0f * m - 1.0f) * 1024.0f; /* fraction scaled to 10 bits, exact */
  uint32_t n = round_half_even_u(q);
  if (n == 1024u) {
    n = 0;
    exp += 1;
  }
  if (exp + 15 >= 31) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | ((uint32_t)(exp + 15) << 10) | n);
}

void oracle_f32_to_f16_array(const float* f, uint16_t* h, int64_t n) {
  for (int64_t i = 0; i < n; ++i) h[i] = oracle_f32_to_f16(f[i]);
}

/* Payload element types: LLMoEBufferLayout<T> with T = bf16, fp16 or fp32. */
#define ORACLE_DT_BF16 0
#define ORACLE_DT_FP16 1
#define ORACLE_DT_FP32 2

static int elem_size(int dt) { return dt == ORACLE_DT_FP32 ? 4 : 2; }

static float load_elem(const uint8_t* p, int dt) {
  if (dt == ORACLE_DT_FP32) {
    float f;
    memcpy(&f, p, 4);
    return f;
  }
  uint16_t b;
  memcpy(&b, p, 2);
  return dt == ORACLE_DT_FP16 ? oracle_f16_to_f32(b) : oracle_bf16_to_f32(b);
}

static void store_elem(uint8_t* p, float v, int dt) {
  if (dt == ORACLE_DT_FP32) {
    memcpy(p, &v, 4);
    return;
  }
  uint16_t b = dt == ORACLE_DT_FP16 ? oracle_f32_to_f16(v) : oracle_f32_to_bf16(v);
  memcpy(p, &b, 2);
}

/* ------------------------------------------------------------------------ */
/* Layout (LL_MoE_Buffers.hpp, LLMoEBufferLayout constructor)               */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint64_t total_bytes;
  uint64_t msg_bytes;             /* sizeof(int) + hidden * sizeof(T) */
  uint64_t send_bytes, recv_bytes, sig_bytes;
  /* byte offsets from the start of one rank's buffer, per set i = 0, 1 */
  uint64_t dispatch_send[2], dispatch_recv[2], dispatch_recv_count[2];
  uint64_t combine_send[2], combine_recv[2], combine_recv_flag[2];
  int64_t num_sig_elems;
} oracle_layout_t;

static int mul_ok(uint64_t a, uint64_t b, uint64_t* r) {
  if (a != 0 && b > UINT64_MAX / a) return 0;
  *r = a * b;
  return 1;
}
static int add_ok(uint64_t a, uint64_t b, uint64_t* r) {
  if (b > UINT64_MAX - a) return 0;
  *r = a + b;
  return 1;
}

/* The constructor's steps in its order.  num_ranks is accepted and unused,
 * as in the header ([[maybe_unused]]).  Returns ORACLE_OK, or ORACLE_BAD_ARG
 * for a dimension below 1, ORACLE_ASSERT where the header's assertion
 * "buffer bytes % sizeof(int) == 0" would fire, ORACLE_OVERFLOW where a
 * product or sum leaves 64 bits. */
int oracle_layout(int num_tokens, int hidden, int num_ranks, int num_experts,
                  int elem_bytes, oracle_layout_t* L) {
  memset(L, 0, sizeof *L);
  if (num_tokens < 1 || hidden < 1 || num_ranks < 1 || num_experts < 1 || elem_bytes < 1)
    return ORACLE_BAD_ARG;
  uint64_t t = (uint64_t)num_tokens, e = (uint64_t)num_experts;
  uint64_t tmp, total = 0;

  /* Message sizes: one int header followed by hidden values of type T; the
   * dispatch and the combine message have the same size. */
  uint64_t dispatch_msg, combine_msg;
  if (!mul_ok((uint64_t)hidden, (uint64_t)elem_bytes, &tmp) || !add_ok(sizeof(int32_t), tmp, &dispatch_msg))
    return ORACLE_OVERFLOW;
  combine_msg = dispatch_msg;

  /* Send buffers: the dispatch sends num_tokens messages, the combine sends
   * num_experts * num_tokens; the region is the larger of the two. */
  uint64_t dispatch_send, combine_send, send;
  if (!mul_ok(t, dispatch_msg, &dispatch_send)) return ORACLE_OVERFLOW;
  if (!mul_ok(e, t, &tmp) || !mul_ok(tmp, combine_msg, &combine_send)) return ORACLE_OVERFLOW;
  send = dispatch_send > combine_send ? dispatch_send : combine_send;
  if (send % sizeof(int32_t) != 0) return ORACLE_ASSERT;
  if (!mul_ok(send, 2, &tmp) || !add_ok(total, tmp, &total)) return ORACLE_OVERFLOW;

  /* Receive buffers: num_experts * num_tokens messages for both roles. */
  uint64_t dispatch_recv, combine_recv, recv;
  if (!mul_ok(e, t, &tmp) || !mul_ok(tmp, dispatch_msg, &dispatch_recv)) return ORACLE_OVERFLOW;
  if (!mul_ok(e, t, &tmp) || !mul_ok(tmp, combine_msg, &combine_recv)) return ORACLE_OVERFLOW;
  recv = dispatch_recv > combine_recv ? dispatch_recv : combine_recv;
  if (recv % sizeof(int32_t) != 0) return ORACLE_ASSERT;
  if (!mul_ok(recv, 2, &tmp) || !add_ok(total, tmp, &total)) return ORACLE_OVERFLOW;

  /* Signaling buffers: one int64 per expert. */
  uint64_t sig = e * sizeof(int64_t);
  if (!mul_ok(sig, 2, &tmp) || !add_ok(total, tmp, &total)) return ORACLE_OVERFLOW;

  /* Pointer assignment: set i's send region after i send regions, its recv
   * region after both send regions and i recv regions, its signal words after
   * both send and both recv regions and i signal regions.  The combine roles
   * reuse the dispatch roles' addresses in the same set. */
  for (int i = 0; i < 2; ++i) {
    uint64_t ii = (uint64_t)i;
    L->dispatch_send[i] = send * ii;
    L->dispatch_recv[i] = send * 2 + recv * ii;
    L->dispatch_recv_count[i] = send * 2 + recv * 2 + sig * ii;
    L->combine_send[i] = send * ii;
    L->combine_recv[i] = send * 2 + recv * ii;
    L->combine_recv_flag[i] = send * 2 + recv * 2 + sig * ii;
  }
  L->total_bytes = total;
  L->msg_bytes = dispatch_msg;
  L->send_bytes = send;
  L->recv_bytes = recv;
  L->sig_bytes = sig;
  L->num_sig_elems = num_experts;
  return ORACLE_OK;
}

/* get_rdma_size_hint: the layout built on a null base, total_bytes returned.
 * 0 when the layout cannot be formed. */
uint64_t oracle_size_hint(int num_max_tokens, int hidden, int num_ranks, int num_experts, int elem_bytes) {
  oracle_layout_t L;
  return oracle_layout(num_max_tokens, hidden, num_ranks, num_experts, elem_bytes, &L) == ORACLE_OK
             ? L.total_bytes : 0;
}

/* ------------------------------------------------------------------------ */
/* Routing count / prefix (the slots and the per-bucket counts)             */
/* ------------------------------------------------------------------------ */

/* Input checks shared by route, dispatch and combine: every id in [-1, E)
 * and no expert twice inside one token. */
static int check_ids(int R, int T, int K, int E, const int64_t* idx) {
  for (int64_t i = 0; i < (int64_t)R * T; ++i) {
    for (int k = 0; k < K; ++k) {
      int64_t e = idx[i * K + k];
      if (e < -1 || e >= E) return ORACLE_BAD_EXPERT;
    }
    for (int k = 0; k < K; ++k)
      for (int k2 = k + 1; k2 < K; ++k2)
        if (idx[i * K + k] >= 0 && idx[i * K + k] == idx[i * K + k2]) return ORACLE_DUPLICATE;
  }
  return ORACLE_OK;
}

/* For every source rank src, every token t of src (ascending) and every top-k
 * position k: if e = idx[src][t][k] is -1 the entry is masked (slot -1);
 * otherwise its slot is the number of earlier tokens t' < t of the same src
 * that chose e, so a bucket (e, src) holds its tokens in ascending token
 * order.  cnt[e * R + src] ends as the number of tokens of src that chose e.
 * Reading: the slot order inside a bucket is ascending source token; the
 * layout header leaves it open.  Returns ORACLE_OK or an input error. */
int oracle_route(int R, int T, int K, int E, const int64_t* idx, int32_t* slot, int64_t* cnt) {
  if (R < 1 || T < 0 || K < 1 || E < 1) return ORACLE_BAD_ARG;
  int rc = check_ids(R, T, K, E, idx);
  if (rc != ORACLE_OK) return rc;
  int64_t* running = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  if (!running) return ORACLE_BAD_ARG;
  for (int src = 0; src < R; ++src) {
    memset(running, 0, (size_t)E * sizeof(int64_t));
    for (int t = 0; t < T; ++t) {
      for (int k = 0; k < K; ++k) {
        int64_t pos = ((int64_t)src * T + t) * K + k;
        int64_t e = idx[pos];
        if (e < 0) {
          slot[pos] = -1;
          continue;
        }
        slot[pos] = (int32_t)running[e];
        running[e] += 1;
      }
    }
    for (int e = 0; e < E; ++e) cnt[(int64_t)e * R + src] = running[e];
  }
  free(running);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Dispatch                                                                  */
/* ------------------------------------------------------------------------ */

/* Expected result of a dispatch into one buffer set, in compact form (only
 * the rows that are written).  Experts are owned in contiguous blocks: with
 * L = E / R local experts per rank, expert e lives on rank dst = e / L as
 * local expert le = e % L.  The unmasked entry (src, t, k) becomes one
 * message [int32 t][x[src][t][0..H) as T] (the int header is read as the
 * source token index; T is bf16, fp16 or fp32, so 4 + H * sizeof(T) bytes) at row (le * R + src) * T_max + slot of rank dst's
 * dispatch receive region, i.e. recv[le][src][slot] with T_max rows per
 * (le, src) pair: the num_experts * num_tokens rows of the header's recv
 * buffer.  Word le * R + src of rank dst's recv-count words receives the
 * bucket's count (a plain count; all R * E words are written).
 *
 * Outputs, n = number of unmasked entries, in (src, t, k) order:
 *   row_rank[n], row_index[n]          where each message goes,
 *   msgs[n][4 + 2H]                     its bytes,
 *   count_words[R][E]                   rank r's E count words.
 * Returns ORACLE_OK or an input error; *n_out receives n. */
int oracle_dispatch(int R, int T_max, int T, int H, int E, int K, int dtype, const uint8_t* x, const int64_t* idx,
                    int64_t* row_rank, int64_t* row_index, uint8_t* msgs, int64_t* count_words,
                    int64_t* n_out) {
  *n_out = 0;
  if (R < 1 || T_max < 1 || T < 0 || T > T_max || H < 1 || E < 1 || K < 1 || E % R != 0) return ORACLE_BAD_ARG;
  int64_t ntk = (int64_t)R * T * K;
  int32_t* slot = (int32_t*)malloc((size_t)(ntk > 0 ? ntk : 1) * sizeof(int32_t));
  int64_t* cnt = (int64_t*)malloc((size_t)E * R * sizeof(int64_t));
  if (!slot || !cnt) {
    free(slot);
    free(cnt);
    return ORACLE_BAD_ARG;
  }
  int rc = oracle_route(R, T, K, E, idx, slot, cnt);
  if (rc != ORACLE_OK) {
    free(slot);
    free(cnt);
    return rc;
  }
  const int L = E / R;
  const size_t row_bytes = (size_t)H * elem_size(dtype);
  const size_t msg = 4 + row_bytes;
  int64_t n = 0;
  for (int src = 0; src < R; ++src) {
    for (int t = 0; t < T; ++t) {
      for (int k = 0; k < K; ++k) {
        int64_t pos = ((int64_t)src * T + t) * K + k;
        int64_t e = idx[pos];
        if (e < 0) continue;
        int dst = (int)(e / L), le = (int)(e % L);
        row_rank[n] = dst;
        row_index[n] = ((int64_t)le * R + src) * T_max + slot[pos];
        uint8_t* out = msgs + (size_t)n * msg;
        int32_t header = t;
        memcpy(out, &header, 4);
        memcpy(out + 4, x + ((size_t)src * T + t) * row_bytes, row_bytes);
        n += 1;
      }
    }
  }
  for (int e = 0; e < E; ++e) {
    for (int src = 0; src < R; ++src) {
      int dst = e / L, le = e % L;
      count_words[(int64_t)dst * E + (int64_t)le * R + src] = cnt[(int64_t)e * R + src];
    }
  }
  *n_out = n;
  free(slot);
  free(cnt);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Combine                                                                   */
/* ------------------------------------------------------------------------ */

/* out[src][t][h] = T_rne( sum over k = 0..K-1 ascending, idx != -1, of
 *                         fl32( w[src][t][k] * f32(y_row[h]) ) )
 * with T the payload type (bf16 or fp16 rounded to nearest even; fp32 kept)
 * where y_row is the expert output for the row that token's entry occupied
 * in the dispatch: the expert outputs are indexed like the receive rows of all
 * ranks laid end to end, row e * R * T_max + src * T_max + slot.  The
 * accumulator starts at +0.0f; each product is rounded to binary32 and then
 * added and rounded (no fused multiply-add); a fully masked token gives +0.0.
 * Masked weights are ignored (no renormalisation).  Rank src's E combine flag
 * words receive, at word e, the number of rows that expert e returns to src.
 *
 * y_rows[E * R * T_max] holds one pointer per expert-output row (H bf16
 * values); rows that no entry uses are never read and may be NULL.
 * Returns ORACLE_OK or an input error. */
int oracle_combine(int R, int T_max, int T, int H, int E, int K, int dtype, const uint8_t* const* y_rows,
                   const int64_t* idx, const float* w, uint8_t* out, int64_t* flag_words) {
  if (R < 1 || T_max < 1 || T < 0 || T > T_max || H < 1 || E < 1 || K < 1 || E % R != 0) return ORACLE_BAD_ARG;
  int64_t ntk = (int64_t)R * T * K;
  int32_t* slot = (int32_t*)malloc((size_t)(ntk > 0 ? ntk : 1) * sizeof(int32_t));
  int64_t* cnt = (int64_t*)malloc((size_t)E * R * sizeof(int64_t));
  float* acc = (float*)malloc((size_t)H * sizeof(float));
  if (!slot || !cnt || !acc) {
    free(slot);
    free(cnt);
    free(acc);
    return ORACLE_BAD_ARG;
  }
  int rc = oracle_route(R, T, K, E, idx, slot, cnt);
  if (rc != ORACLE_OK) {
    free(slot);
    free(cnt);
    free(acc);
    return rc;
  }
  const size_t es = (size_t)elem_size(dtype);
  for (int src = 0; src < R; ++src) {
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < H; ++h) acc[h] = 0.0f;
      for (int k = 0; k < K; ++k) {
        int64_t pos = ((int64_t)src * T + t) * K + k;
        int64_t e = idx[pos];
        if (e < 0) continue;
        int64_t row = e * R * T_max + (int64_t)src * T_max + slot[pos];
        const uint8_t* y = y_rows[row];
        float wk = w[pos];
        for (int h = 0; h < H; ++h) {
          float p = wk * load_elem(y + (size_t)h * es, dtype);
          acc[h] = acc[h] + p;
        }
      }
      uint8_t* o = out + ((size_t)src * T + t) * H * es;
      for (int h = 0; h < H; ++h) store_elem(o + (size_t)h * es, acc[h], dtype);
    }
  }
  for (int src = 0; src < R; ++src)
    for (int e = 0; e < E; ++e) flag_words[(int64_t)src * E + e] = cnt[(int64_t)e * R + src];
  free(slot);
  free(cnt);
  free(acc);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Clean (LLMoEBuffer::clean_meta)                                           */
/* ------------------------------------------------------------------------ */

/* clean_meta() hands back the set's recv-count pointer (equal to its combine
 * recv-flag pointer) and num_sig_elems = num_experts: the clean zeroes those
 * E int64 words, here on every one of the R ranks. */
void oracle_clean(int R, int E, int64_t* sig_words) {
  for (int64_t i = 0; i < (int64_t)R * E; ++i) sig_words[i] = 0;
}

/* ------------------------------------------------------------------------ */
/* Staged combine (LLMoEBuffer combine send / recv roles)                   */
/* ------------------------------------------------------------------------ */

/* The combine routed through the combine receive buffers.  Step one: every
 * unmasked entry (src, t, k) choosing expert e has its expert output row
 * returned to rank src as one message [int32 t][y_row as T] at row
 * e * T_max + t of rank src's combine receive region (combine_recv[e][t]: the
 * num_experts * num_tokens messages the layout sizes that buffer for).
 * Step two: rank src reduces out[src][t] from the payloads of its messages
 * combine_recv[e_k][t], over ascending k, with the arithmetic of
 * oracle_combine.  Flag word e of rank src = rows expert e returned to src.
 *
 * Outputs: msg_rank[n], msg_row[n], msgs[n][4 + 2H] in (src, t, k) order of
 * the unmasked entries, out[R][T][H], flag_words[R][E].  *n_out = n. */
int oracle_combine_staged(int R, int T_max, int T, int H, int E, int K, int dtype, const uint8_t* const* y_rows,
                          const int64_t* idx, const float* w, int64_t* msg_rank, int64_t* msg_row, uint8_t* msgs,
                          uint8_t* out, int64_t* flag_words, int64_t* n_out) {
  *n_out = 0;
  if (R < 1 || T_max < 1 || T < 0 || T > T_max || H < 1 || E < 1 || K < 1 || E % R != 0) return ORACLE_BAD_ARG;
  int64_t ntk = (int64_t)R * T * K;
  int32_t* slot = (int32_t*)malloc((size_t)(ntk > 0 ? ntk : 1) * sizeof(int32_t));
  int64_t* cnt = (int64_t*)malloc((size_t)E * R * sizeof(int64_t));
  int64_t* where = (int64_t*)malloc((size_t)(ntk > 0 ? ntk : 1) * sizeof(int64_t));
  float* acc = (float*)malloc((size_t)H * sizeof(float));
  if (!slot || !cnt || !where || !acc) {
    free(slot); free(cnt); free(where); free(acc);
    return ORACLE_BAD_ARG;
  }
  int rc = oracle_route(R, T, K, E, idx, slot, cnt);
  if (rc != ORACLE_OK) {
    free(slot); free(cnt); free(where); free(acc);
    return rc;
  }
  const size_t es = (size_t)elem_size(dtype);
  const size_t msg = 4 + (size_t)H * es;
  /* step one: the returned messages */
  int64_t n = 0;
  for (int src = 0; src < R; ++src) {
    for (int t = 0; t < T; ++t) {
      for (int k = 0; k < K; ++k) {
        int64_t pos = ((int64_t)src * T + t) * K + k;
        int64_t e = idx[pos];
        where[pos] = -1;
        if (e < 0) continue;
        int64_t yrow = e * R * T_max + (int64_t)src * T_max + slot[pos];
        msg_rank[n] = src;
        msg_row[n] = e * T_max + t;
        uint8_t* m = msgs + (size_t)n * msg;
        int32_t header = t;
        memcpy(m, &header, 4);
        memcpy(m + 4, y_rows[yrow], (size_t)H * es);
        where[pos] = n;
        n += 1;
      }
    }
  }
  /* step two: each source rank reduces from its received messages */
  for (int src = 0; src < R; ++src) {
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < H; ++h) acc[h] = 0.0f;
      for (int k = 0; k < K; ++k) {
        int64_t pos = ((int64_t)src * T + t) * K + k;
        if (where[pos] < 0) continue;
        const uint8_t* payload = msgs + (size_t)where[pos] * msg + 4;
        float wk = w[pos];
        for (int h = 0; h < H; ++h) {
          float p = wk * load_elem(payload + (size_t)h * es, dtype);
          acc[h] = acc[h] + p;
        }
      }
      uint8_t* o = out + ((size_t)src * T + t) * H * es;
      for (int h = 0; h < H; ++h) store_elem(o + (size_t)h * es, acc[h], dtype);
    }
  }
  for (int src = 0; src < R; ++src)
    for (int e = 0; e < E; ++e) flag_words[(int64_t)src * E + e] = cnt[(int64_t)e * R + src];
  *n_out = n;
  free(slot); free(cnt); free(where); free(acc);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Unpack: the received messages as the experts' input                      */
/* ------------------------------------------------------------------------ */

/* The experts' view of a dispatch: for every unmasked entry (src, t, k)
 * choosing expert e, its token row x[src][t] at row e * R * T_max +
 * src * T_max + slot of recv_x (for rank dst = e / L and local expert
 * le = e % L that is recv_x[dst][le][src * T_max + slot]: the receive rows
 * of each local expert laid out contiguously, the same order the combine
 * reads its expert outputs in), and the token index t at the same position
 * of recv_src.  Rows no entry reaches are not written.  Returns the number of
 * rows written in *n_out and, in rows[n], which rows they are, in (src, t, k)
 * order. */
int oracle_unpack(int R, int T_max, int T, int H, int E, int K, int dtype, const uint8_t* x, const int64_t* idx,
                  uint8_t* recv_x, int32_t* recv_src, int64_t* rows, int64_t* n_out) {
  *n_out = 0;
  if (R < 1 || T_max < 1 || T < 0 || T > T_max || H < 1 || E < 1 || K < 1 || E % R != 0) return ORACLE_BAD_ARG;
  int64_t ntk = (int64_t)R * T * K;
  int32_t* slot = (int32_t*)malloc((size_t)(ntk > 0 ? ntk : 1) * sizeof(int32_t));
  int64_t* cnt = (int64_t*)malloc((size_t)E * R * sizeof(int64_t));
  if (!slot || !cnt) {
    free(slot);
    free(cnt);
    return ORACLE_BAD_ARG;
  }
  int rc = oracle_route(R, T, K, E, idx, slot, cnt);
  if (rc != ORACLE_OK) {
    free(slot);
    free(cnt);
    return rc;
  }
  const size_t row_bytes = (size_t)H * elem_size(dtype);
  int64_t n = 0;
  for (int src = 0; src < R; ++src)
    for (int t = 0; t < T; ++t)
      for (int k = 0; k < K; ++k) {
        int64_t pos = ((int64_t)src * T + t) * K + k;
        int64_t e = idx[pos];
        if (e < 0) continue;
        int64_t row = e * R * T_max + (int64_t)src * T_max + slot[pos];
        memcpy(recv_x + (size_t)row * row_bytes, x + ((size_t)src * T + t) * row_bytes, row_bytes);
        recv_src[row] = t;
        rows[n++] = row;
      }
  *n_out = n;
  free(slot);
  free(cnt);
  return ORACLE_OK;
}
