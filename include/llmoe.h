/*
 * llmoe.h -- C ABI of the GB300 (sm_103a) low-latency MoE dispatch / combine
 * library (libllmoe.so).
 *
 * One GPU holds R simulated expert-parallel ranks as R disjoint segments of
 * one device allocation ("rank buffers").  Each rank buffer has the layout of
 * LLMoEBufferLayout<T> from LL_MoE_Buffers.hpp (rocshmem LL_MoE example) for
 * a payload type T of bf16 (the default), fp16 or fp32: two buffer sets, each
 * with a send region, a receive region and num_experts int64 signal words;
 * the combine roles alias the dispatch roles of the same set.  Messages are
 * one int32 header (the source token index) followed by `hidden` values of
 * type T, 4 + hidden * sizeof(T) bytes, packed without padding.
 *
 * Conventions for every call:
 *   - All pointers passed to the data-path calls are DEVICE pointers into
 *     memory the caller allocated; the library never allocates, frees or
 *     synchronises (except llmoe_get_error, which reads a word back).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and runs asynchronously; buffers must stay alive until it ends.
 *   - A call returns LLMOE_SUCCESS once its kernel is enqueued.  Argument
 *     checks are done on the host before any launch: a call that returns
 *     LLMOE_ERR_INVALID_ARGUMENT or LLMOE_ERR_INVALID_USAGE launched nothing.
 *     LLMOE_ERR_CUDA reports a launch error (cudaGetLastError).
 *   - Payload values (x, y, out) are of the set's payload type T (bf16 by
 *     default; fp16 or fp32 through llmoe_buf_set_t.dtype).
 *
 * Sequencing: a set's signal words must be zero before a dispatch or combine
 * writes them (llmoe_clean zeroes them).  A round alternates sets:
 *   llmoe_clean(set 0); llmoe_dispatch(set 0); llmoe_clean(set 1);
 *   llmoe_combine(set 1)
 * so a combine never overwrites counts that consumers of the dispatch read.
 */
#ifndef LLMOE_H_
#define LLMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols keep default visibility when the library is built with
 * -fvisibility=hidden. */
#if defined(__GNUC__)
#define LLMOE_API __attribute__((visibility("default")))
#else
#define LLMOE_API
#endif

/* A cudaStream_t without including the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* llmoe_stream_t;

/* Status codes.  The values follow mscclpp.h's mscclppResult_t (Success 0,
 * UnhandledCudaError 1, InvalidArgument 4, InvalidUsage 5). */
typedef enum {
  LLMOE_SUCCESS = 0,
  LLMOE_ERR_CUDA = 1,
  LLMOE_ERR_INVALID_ARGUMENT = 4,
  LLMOE_ERR_INVALID_USAGE = 5
} llmoe_status_t;

/* Device error-word codes, written only when llmoe_buf_set_t.err is non-NULL
 * (validate mode); the first error a launch meets wins.  Like the refusal
 * words of memra-engine tp_ar.rs (barrier_errors), the word is read back
 * with llmoe_get_error, which drains the stream, so it belongs in tests and
 * gates, not in the hot loop. */
#define LLMOE_DEV_OK 0
#define LLMOE_DEV_BAD_EXPERT 1   /* a top-k id outside [-1, num_experts) */
#define LLMOE_DEV_DUPLICATE 2    /* one expert twice in one token's top-k */
#define LLMOE_DEV_STALE_SIGNAL 3 /* a signal word was non-zero on entry (a clean was skipped) */
#define LLMOE_DEV_SLOT_RANGE 4   /* a bucket overflowed num_max_tokens (only reachable with duplicates) */
#define LLMOE_DEV_TIMEOUT 5      /* a bounded wait inside a kernel expired (a copy never completed, or a
                                    signal word was never raised) */
#define LLMOE_DEV_BAD_MESSAGE 6  /* a staged-combine message header does not name its token */

/* llmoe_buf_set_t.flags */
/* The call's read-only routing inputs (topk_idx and topk_w, and x for a
 * dispatch) were complete before the kernel that precedes this call on the
 * stream started, so the call's kernel may read them (and run its routing
 * scan) while that kernel drains.  The expert outputs y of a combine, the
 * rank buffers and the output are never touched before the preceding kernel
 * has completed.  Typical use: a combine whose topk_idx / topk_w came from a
 * router that ran before the expert kernels. */
#define LLMOE_FLAG_INPUTS_READY 1u
/* A dispatch or combine on set s also zeroes set s^1's num_experts signal
 * words in every rank buffer (the llmoe_clean that the next call on set s^1
 * needs), after the preceding kernel on the stream has completed.  A round
 * then needs two launches: dispatch(set 0) and combine(set 1), each with this
 * flag, after one llmoe_clean of set 0 before the first round.  Whatever
 * reads the other set's words must do so before this call. */
#define LLMOE_FLAG_CLEAN_OTHER_SET 2u

/* llmoe_buf_set_t.dtype: the payload type T of LLMoEBufferLayout<T>.  A
 * message is 4 + hidden * sizeof(T) bytes; hidden * sizeof(T) must be a
 * multiple of 16.  The combine accumulates in fp32 and stores T (bf16 and
 * fp16 rounded to nearest even, fp32 as accumulated). */
#define LLMOE_DTYPE_BF16 0
#define LLMOE_DTYPE_FP16 1
#define LLMOE_DTYPE_FP32 2

/* Library limits (checked on the host). */
#define LLMOE_MAX_TOPK 32
#define LLMOE_MAX_EXPERTS 8192

/* One buffer set of the R rank buffers, plus the geometry of one call.
 *   base           device pointer, 16-byte aligned; rank r's buffer starts at
 *                  base + r * rank_stride.
 *   rank_stride    bytes between rank buffers; a multiple of 16 and at least
 *                  llmoe_layout_bytes(num_max_tokens, hidden, num_ranks,
 *                  num_experts).
 *   num_max_tokens T: tokens per rank the layout was sized for (the worst-case
 *                  micro-batch; "num_max_dispatch_tokens_per_rank").
 *   num_tokens     tokens per rank in this call, 0 <= num_tokens <= T.
 *   hidden         H, values per token; H * sizeof(T) a multiple of 16.
 *   num_ranks      R >= 1.
 *   num_experts    E, a multiple of R, <= LLMOE_MAX_EXPERTS.  Expert e is
 *                  owned by rank e / (E/R) as local expert e % (E/R).
 *   num_topk       K, 1 <= K <= min(E, LLMOE_MAX_TOPK).
 *   set            0 or 1: which of the layout's two buffer sets.
 *   err            optional device int32 word; NULL turns validation off.
 *                  With validation off, invalid ids are still skipped and no
 *                  access leaves the buffers, but nothing is reported.
 *   flags          LLMOE_FLAG_* bits; 0 for the plain stream order.
 *   dtype          LLMOE_DTYPE_*: the payload type (0 = bf16). */
typedef struct {
  void* base;
  uint64_t rank_stride;
  int32_t num_max_tokens;
  int32_t num_tokens;
  int32_t hidden;
  int32_t num_ranks;
  int32_t num_experts;
  int32_t num_topk;
  int32_t set;
  int32_t* err;
  uint32_t flags;
  int32_t dtype;
} llmoe_buf_set_t;

/* Bytes of ONE rank buffer: get_rdma_size_hint<bf16>(num_max_tokens, hidden,
 * num_ranks, num_experts) of LL_MoE_Buffers.hpp, i.e. LLMoEBufferLayout's
 * total_bytes = 2 * max(send) + 2 * max(recv) + 2 * 8 * num_experts.
 * num_ranks does not change the size (it is [[maybe_unused]] there).
 * Returns 0 when a dimension is < 1, when the layout's "bytes %
 * sizeof(int) == 0" assertion would fail, or when a size overflows 64 bits.
 * Host only; touches no device. */
LLMOE_API size_t llmoe_layout_bytes(int num_max_tokens, int hidden, int num_ranks, int num_experts);

/* The same for payload type `dtype` (LLMOE_DTYPE_*): get_rdma_size_hint<T>. */
LLMOE_API size_t llmoe_layout_bytes_dtype(int num_max_tokens, int hidden, int num_ranks, int num_experts, int dtype);

/* Byte offsets, from the start of a rank buffer, of buffer set `set`'s send
 * region, receive region and signal words (LLMoEBufferLayout, "Assign
 * pointers"; the combine send / recv / flag of a set are the same addresses
 * as its dispatch send / recv / count).  Any output pointer may be NULL.
 * Returns LLMOE_SUCCESS, or LLMOE_ERR_INVALID_ARGUMENT when
 * llmoe_layout_bytes would return 0 or set is not 0 or 1. */
LLMOE_API int llmoe_layout_offsets(int num_max_tokens, int hidden, int num_ranks, int num_experts, int set,
                         uint64_t* send_offset, uint64_t* recv_offset, uint64_t* signal_offset);

/* The same for payload type `dtype` (LLMOE_DTYPE_*). */
LLMOE_API int llmoe_layout_offsets_dtype(int num_max_tokens, int hidden, int num_ranks, int num_experts, int dtype,
                                         int set, uint64_t* send_offset, uint64_t* recv_offset,
                                         uint64_t* signal_offset);

/* Routing count / prefix scan, on its own (dispatch and combine run the same
 * scan inside their kernels and do not need this call).
 *   topk_idx  device int64 [R][num_tokens][K], -1 = masked.
 *   slot      device int32 [R][num_tokens][K] out: for an unmasked entry
 *             (src, t, k) choosing expert e, the number of earlier tokens
 *             t' < t of src that chose e (ascending source-token order inside
 *             each (expert, source) bucket); -1 where masked or invalid.
 *   counts    device int64 [E][R] out: tokens of src that chose e.
 * Only the geometry fields of `bs` are used (base / rank_stride / set are not
 * read and may be zero); err as for the other calls. */
LLMOE_API int llmoe_route(const int64_t* topk_idx, int32_t* slot, int64_t* counts, const llmoe_buf_set_t* bs,
                llmoe_stream_t stream);

/* Dispatch (LLMoEBuffer dispatch receive buffer and recv-count words).
 *   x         device T [R][num_tokens][H] (T per bs->dtype), 16-byte aligned.
 *   topk_idx  device int64 [R][num_tokens][K], -1 = masked.
 * For every unmasked entry (src, t, k) choosing expert e, owned by rank
 * dst = e / L as local expert le = e % L, writes the message
 * [int32 t][x[src][t][0..H)] at row (le * R + src) * T + slot of rank dst's
 * set-`set` receive region (recv[le][src][slot]), slot as in llmoe_route.
 * Then writes rank dst's signal word le * R + src = that bucket's count, for
 * all R * E words.  Nothing else is written: unused receive rows keep their
 * contents. */
LLMOE_API int llmoe_dispatch(const void* x, const int64_t* topk_idx, const llmoe_buf_set_t* bs,
                   llmoe_stream_t stream);

/* Combine (LLMoEBuffer combine roles; the expert outputs are gathered in
 * place instead of being staged through the combine send / recv regions).
 *   y         device T [E * R * T][H], 16-byte aligned: the expert
 *             outputs in receive-row order, row e * R * T + src * T + slot
 *             for the entry that occupied recv[le][src][slot] of rank e / L.
 *   topk_idx  device int64 [R][num_tokens][K], -1 = masked.
 *   topk_w    device fp32 [R][num_tokens][K].
 *   out       device T [R][num_tokens][H] out, 16-byte aligned;
 *             must not overlap y.
 * out[src][t][:] = T(sum over ascending k of unmasked entries of
 * fl32(w * fp32(y_row))), starting from +0.0, each product rounded to fp32
 * before it is added (no fused multiply-add); T() rounds to nearest even for
 * bf16 / fp16.  Then writes rank src's
 * set-`set` signal word e = number of rows expert e returned to src. */
LLMOE_API int llmoe_combine(const void* y, const int64_t* topk_idx, const float* topk_w, void* out,
                  const llmoe_buf_set_t* bs, llmoe_stream_t stream);

/* Staged combine (LLMoEBuffer combine receive buffer and recv-flag words): the
 * same inputs and result as llmoe_combine, routed through the layout's
 * combine buffers as the expert-parallel exchange would route it.  First, for
 * every unmasked entry (src, t, k) choosing expert e, the expert output row
 * returns to rank src as the message [int32 t][y row] at row e * T + t of
 * rank src's set-`set` receive region (combine_recv[e][t]: the
 * num_experts * num_tokens messages of the combine receive buffer), and rank
 * src's flag word e is set to the rows e returned.  Then rank src reduces
 * out[src][t] from those messages' payloads exactly as llmoe_combine does
 * (ascending k, fp32 products then sums, bf16 round-to-nearest-even).  Two
 * kernels; the second starts after the first has completed.  Validate mode
 * also checks each message header (LLMOE_DEV_BAD_MESSAGE).  The set's receive
 * region is overwritten at those rows: it aliases the dispatch receive region
 * of the same set. */
LLMOE_API int llmoe_combine_staged(const void* y, const int64_t* topk_idx, const float* topk_w, void* out,
                                   const llmoe_buf_set_t* bs, llmoe_stream_t stream);

/* Unpack: the experts' view of a completed dispatch on set `set`.  For every
 * rank dst, local expert le and source rank src, reads the bucket's count
 * (rank dst's signal word le * R + src) and its messages
 * recv[le][src][0..count), and writes each message's payload to row
 * (dst * L + le) * R * T + src * T + slot of recv_x and its header (the source
 * token index) to the same position of recv_src.  recv_x [E * R * T][H] of the
 * payload type (16-byte aligned) thus holds each local expert's received rows
 * contiguously, in the order llmoe_combine reads its expert outputs y;
 * recv_src is int32 [E * R * T].  Rows past a bucket's count are not written.
 * Uses no routing input: the counts in the rank buffers drive it. */
LLMOE_API int llmoe_unpack(void* recv_x, int32_t* recv_src, const llmoe_buf_set_t* bs, llmoe_stream_t stream);

/* Dispatch with the experts' input rows: the messages and recv-count words of
 * llmoe_dispatch, and in the same launch the recv_x rows and recv_src words
 * that llmoe_unpack would make from them (same layout and rows; rows past a
 * bucket's count are not written).  The CTA that moves a token holds its row
 * and knows its slots, so it writes each row straight to recv_x beside the
 * message, and no message is read back.  The result equals llmoe_dispatch
 * followed by llmoe_unpack.  recv_x and recv_src as for llmoe_unpack (16- and
 * 4-byte aligned, not NULL); they must not overlap the rank buffers, x or
 * topk_idx.  Flags as for llmoe_dispatch. */
LLMOE_API int llmoe_dispatch_unpack(const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src,
                                    const llmoe_buf_set_t* bs, llmoe_stream_t stream);

/* Bytes of the workspace llmoe_dispatch_signaled needs for this geometry.
 * No counterpart in the layout header: it holds one completion counter per
 * source rank (producers) and one for the consumers. */
LLMOE_API size_t llmoe_signal_workspace_bytes(const llmoe_buf_set_t* bs);

/* Dispatch and unpack in one cooperative launch whose CTAs signal each other
 * through the recv-count words, the way the expert-parallel exchange signals
 * a receiving rank (one-sided put, then signal; the receiver reads only after
 * its wait returns: mscclpp.h, mscclppDevConn put / signal / wait).
 * Producer work is the dispatch of llmoe_dispatch.  When every CTA of a
 * source rank has written its rows, the last one writes that source's
 * signal words as -(count + 1).  Consumer work runs on the same CTAs, its
 * warps grouped by source rank: a warp of source s waits for every signal
 * word of s to become non-zero, then unpacks an equal share of s's received
 * rows as llmoe_unpack does.  The last warp to finish rewrites every raised
 * word to the plain count.  The result is that of llmoe_dispatch followed by
 * llmoe_unpack.
 *   workspace   device memory of llmoe_signal_workspace_bytes(bs) bytes,
 *               zero before the first call; each completed call leaves it
 *               zero.  After an LLMOE_DEV_TIMEOUT, zero it again.
 *   spin_limit  clock cycles a consumer waits for one signal word before it
 *               records LLMOE_DEV_TIMEOUT (needs bs->err) and skips that
 *               source; about 2e9 is one second at 2 GHz.  Unlike the
 *               unbounded waits of mscclpp.h, no wait here can hang.
 * Returns LLMOE_ERR_INVALID_ARGUMENT when the grid this geometry needs cannot
 * be resident all at once (the signalling needs every CTA running). */
LLMOE_API int llmoe_dispatch_signaled(const void* x, const int64_t* topk_idx, void* recv_x, int32_t* recv_src,
                                      void* workspace, int64_t spin_limit, const llmoe_buf_set_t* bs,
                                      llmoe_stream_t stream);

/* Largest num_ranks llmoe_dispatch_signaled_static accepts. */
#define LLMOE_STATIC_MAX_RANKS 1024

/* llmoe_dispatch_signaled for callers that cannot allocate device memory.
 * The pages have no counterpart for this call.
 * Some callers have no way to obtain scratch memory at the point of the
 * call: a plugin handed only raw device pointers by a host framework that
 * owns every allocation, or a latency-critical loop in which a cudaMalloc,
 * which may synchronize the device, is not acceptable.  This call needs no
 * workspace from them: the completion counters (one per source, one for the
 * consumers) live in a fixed device array inside the library, sized for
 * LLMOE_STATIC_MAX_RANKS ranks (about 4 KB, held by every GPU that loads the
 * library until the process exits).
 * It allocates nothing and calls no allocating routine.
 *   - Same arguments and result as llmoe_dispatch_signaled, minus the
 *     workspace.  num_ranks above LLMOE_STATIC_MAX_RANKS returns
 *     LLMOE_ERR_INVALID_ARGUMENT without launching.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     life of the process; make that first call before any stream capture,
 *     and make no call on a device after a cudaDeviceReset of it (the
 *     array may then sit at another address).
 *   - Every argument check comes first: a call that returns an error has
 *     queued nothing and left the array alone.
 *   - Each call clears the counters it uses (a cudaMemsetAsync on `stream`)
 *     before its kernel.  A launch returns them to zero itself, timed out
 *     or not; the clear covers a launch that never finished.
 *   - All calls on a device share the one array: calls whose kernels
 *     overlap on the GPU (on different streams) race on it and must not be
 *     issued that way. */
LLMOE_API int llmoe_dispatch_signaled_static(const void* x, const int64_t* topk_idx, void* recv_x,
                                             int32_t* recv_src, int64_t spin_limit, const llmoe_buf_set_t* bs,
                                             llmoe_stream_t stream);

/* Clean (LLMoEBuffer::clean_meta): zero the num_experts int64 signal words
 * of buffer set `set` in each of the R rank buffers.  This resets both the
 * dispatch recv counts and the combine recv flags, which share the words. */
LLMOE_API int llmoe_clean(const llmoe_buf_set_t* bs, llmoe_stream_t stream);

/* Validate-mode read-back: waits for `stream`, copies *bs->err into *code
 * (LLMOE_DEV_*) and, if `reset` is non-zero, zeroes the word.  Returns
 * LLMOE_ERR_INVALID_USAGE when bs->err is NULL. */
LLMOE_API int llmoe_get_error(const llmoe_buf_set_t* bs, llmoe_stream_t stream, int32_t* code, int reset);

/* A static string for a status code. */
LLMOE_API const char* llmoe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* LLMOE_H_ */
