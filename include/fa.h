/*
 * fa.h — C ABI of the exact tiled attention library (libfa.so, sm_103a).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale · Q Kᵀ) V        (row-wise softmax, optional causal mask)
 *
 * tile by tile with online softmax, so the N×N score matrix S and the
 * probability matrix P never reach device memory, and its gradient by
 * recomputing each P tile from the saved per-row log-sum-exp.
 *
 * Where the operation is defined:
 *   - attention itself: dcwnkz.com GPU-tricks article (CS336 tricks),
 *     FlashAttention section, "先简要回顾注意力机制" (scores are q·k dot
 *     products; softmax makes each row sum to 1; output = weighted sum of V);
 *   - tiling + online softmax + recomputation: CMU 10-423 L17–L18 notes
 *     (quidproquo.cc), sections 前置二：online softmax and FlashAttention 本身;
 *   - the six-score block-by-block rescaling walk-through: dcwnkz.com
 *     article, FlashAttention section;
 *   - the [B, heads, S, head_dim] layout and the causal mask:
 *     "07-16 下午：分布式大模型训练与推理" (docs.bfyes.cn), section
 *     自回归语言模型推理.
 * The 1/sqrt(d) factor is not printed on those pages; callers pass `scale`.
 *
 * Conventions shared by every entry point
 *   Tensors   q, k, v, o, dO, dq, dk, dv: bf16, contiguous, row-major
 *             [B][H][N][d]; d must be 64 or 128. lse, D: fp32 [B][H][N].
 *             The _gqa forms (and the backward stages) take k, v, dk, dv as
 *             [B][Hkv][N][d] (see fa_fwd_gqa).
 *   Pointers  device pointers, each 16-byte aligned. The caller owns every
 *             buffer; the library allocates no memory, never synchronises
 *             the stream (except fa_last_device_error), and launches on
 *             `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *             stream). Calls are asynchronous: a 0 return means the work was
 *             enqueued.
 *   Outputs   fully overwritten, never accumulated into.
 *   Errors    arguments are checked before anything is launched; on error
 *             nothing is launched and a non-zero fa_status is returned.
 *             Device-side failures (a pipeline wait that exceeded its time
 *             limit) are reported by fa_last_device_error.
 *   Threads   entry points may be called from several host threads; each
 *             call works on its own descriptors.
 *   Devices   per-device state the library keeps (its side streams) lives
 *             as long as the process; after cudaDeviceReset on a device, do
 *             not call into the library on that device again in the same
 *             process.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, B/H/N < 1, Hkv not dividing H, bad scale */
  FA_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, or sizes past 2^31 elements */
  FA_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch error) */
  FA_ERR_TIMEOUT = 5,     /* device pipeline wait exceeded its limit */
  FA_ERR_WORKSPACE = 6,   /* workspace pointer null or smaller than required */
  FA_ERR_BAD_INDEX = 7,   /* (device) a block-table entry outside [0, num_blocks) */
  FA_ERR_BOUNDS = 8       /* (device, FA_DEBUG build) a computed address left its buffer */
} fa_status;

/*
 * Forward pass.
 *   q, k, v  [B][H][N][d] bf16 inputs.
 *   o        [B][H][N][d] bf16 output: softmax(scale·q kᵀ [+ causal mask]) v.
 *   lse      [B][H][N] fp32 output: per-row log-sum-exp of the scaled,
 *            masked scores, natural log: lse_i = ln Σ_j exp(scale·q_i·k_j).
 *   causal   non-zero: query i attends to keys j <= i (top-left aligned).
 * Returns an fa_status.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, void* stream);

/*
 * Grouped-query attention forward. k and v hold Hkv heads, [B][Hkv][N][d];
 * q, o and lse keep H heads. Query head h attends with K/V head h / (H/Hkv):
 * H/Hkv consecutive query heads share one K/V head. ("07-16 下午" notes,
 * section 自回归语言模型推理, Prefill、Decode 与推理调度: with grouped-query
 * attention kv_heads is smaller than the number of query heads, which
 * shrinks the KV cache; the pages give no head mapping, and consecutive
 * groups are the usual one.) Hkv must be >= 1 and divide H, else
 * FA_ERR_INVALID_ARG. fa_fwd is this call with Hkv = H.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Hkv, int N, int d, float scale, int causal, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: the fp32 row vector D [B][H][N]
 * (D_i = Σ_c dO_ic · O_ic). Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass: gradients of o = softmax(scale·q kᵀ) v with respect to q,
 * k, v for the output gradient dO. P is rebuilt tile by tile from q, k and
 * the forward's lse (recomputation), never read from memory.
 *   q, k, v, o, dO  [B][H][N][d] bf16 (o and lse from fa_fwd on q, k, v).
 *   dq, dk, dv      [B][H][N][d] bf16 outputs.
 *   workspace       device buffer of at least fa_bwd_workspace_bytes(...)
 *                   bytes, 16-byte aligned; contents on entry are ignored.
 * Launches the kernels in one of two orders, chosen by fa_bwd_fuses_d:
 *   fused      the dQ sweep, which also forms D (fa_bwd_dq_d), then the
 *              dK/dV sweep, both on `stream`;
 *   side by    preprocess (D) on `stream`, then the dK/dV sweep over query
 *   side       tiles on `stream` and, beside it, the dQ sweep over key tiles
 *              on a side stream the library forks from `stream` after the
 *              preprocess and joins back to it.
 * Work queued on `stream` afterwards sees every kernel; the call is
 * capturable into a CUDA graph. The first call on a host thread and device
 * that takes the side stream creates it, kept until the thread exits. Calls
 * from one host thread share it, so their dQ sweeps run in call order even
 * when the calls are on different streams. The two orders compute D in a
 * different summation order, so their gradients can differ in the last bit
 * of bf16 (both are within the same tolerance of the exact result).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
           int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Grouped-query attention backward (head mapping and Hkv rules as in
 * fa_fwd_gqa). k, v, dk, dv are [B][Hkv][N][d]; dk and dv of a K/V head sum
 * the gradients of every query head that shares it (the dK/dV sweep of one
 * K/V head runs over all query tiles of its H/Hkv query heads, so the sum
 * stays in fp32 on chip and needs no atomics). Workspace as for fa_bwd
 * (fa_bwd_workspace_bytes(B, H, N, d): D has one entry per query row).
 * fa_bwd is this call with Hkv = H.
 */
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
               const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
               int B, int H, int Hkv, int N, int d, float scale, int causal, void* stream);

/*
 * The backward stages as separate calls, each on `stream` (fa_bwd_gqa runs
 * preprocess, dK/dV and dQ, or dQ-with-D then dK/dV: see fa_bwd). They
 * share fa_bwd_gqa's argument rules (Hkv = H for plain multi-head
 * attention); `Dvec` is fp32 [B][H][N] caller-owned device memory.
 *   fa_bwd_preprocess : Dvec_i = Σ_c dO_ic·O_ic.
 *   fa_bwd_dkdv       : dk = scale·dSᵀ q and dv = Pᵀ dO (bf16, final); reads Dvec.
 *   fa_bwd_dq         : dq = scale·dS k (bf16, final); reads Dvec.
 *   fa_bwd_dq_d       : fa_bwd_dq that forms Dvec_i itself from o (loaded
 *                       beside q and dO, one query tile per CTA) and writes
 *                       it, so no preprocess runs; fa_bwd_dkdv goes after it.
 *                       Errors: as fa_bwd_dq, and o NULL or misaligned.
 * fa_bwd_fuses_d returns 1 when fa_bwd_gqa takes the fused order for these
 * sizes on the current device (one K/V head per query head, and a dK/dV grid
 * of at least 4 CTAs per SM), else 0 (also for invalid sizes).
 */
int fa_bwd_preprocess(const void* o, const void* dO, float* Dvec, int B, int H, int N, int d,
                      void* stream);
int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                const float* Dvec, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                float scale, int causal, void* stream);
int fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
              const float* Dvec, void* dq, int B, int H, int Hkv, int N, int d, float scale,
              int causal, void* stream);
int fa_bwd_dq_d(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                float* Dvec, void* dq, int B, int H, int Hkv, int N, int d, float scale, int causal,
                void* stream);
int fa_bwd_fuses_d(int B, int H, int Hkv, int N, int d);

/*
 * Addresses of one attention problem's tensors, in host or in device
 * memory depending on the argument they are passed as. Shapes and types as
 * in fa_fwd_gqa / fa_bwd_gqa: q, dO, o, dq [B][H][N][d] bf16; k, v, dk, dv
 * [B][Hkv][N][d] bf16; lse [B][H][N] fp32. dO, dq, dk, dv are unused (may
 * be NULL) in fa_fwd_host.
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* dO;
  void* o;
  float* lse;
  void* dq;
  void* dk;
  void* dv;
} fa_tensors;

/*
 * Attention from host memory: copies q, k, v (and dO) from `host` to the
 * device buffers in `dev`, runs fa_fwd_gqa (and fa_bwd_gqa, its D vector
 * in `workspace`, fa_bwd_workspace_bytes(B, H, N, d) bytes) on them, and
 * copies o, lse (and dq, dk, dv) back into `host`. The results are those
 * of the device calls, bit for bit, and are also left in `dev`.
 *
 * The (batch, K/V head) pairs are independent problems, so the work is cut
 * into n_chunks slices of consecutive pairs (more than B·Hkv or 64 is
 * clamped; 0 lets the library choose: up to 8, as long as each slice's
 * dK/dV sweep keeps 1.5 CTAs per SM), and each slice's copies overlap
 * other slices' kernels: its
 * inputs go in on a copy-in stream, its kernels run on `stream`, its
 * outputs come out on a copy-out stream as soon as they are ready. Host
 * buffers should be page-locked (cudaHostAlloc / cudaHostRegister), else
 * the CUDA driver stages the copies and they do not overlap.
 *
 *   Ordering   the call starts after the work already queued on `stream`,
 *              and work queued on `stream` after it starts after every
 *              copy of this call has finished: synchronise `stream`
 *              before reading the host outputs or reusing the host inputs.
 *   Resources  the first call on a host thread and device creates two
 *              non-blocking CUDA streams, kept until the thread exits;
 *              each call creates and releases a few CUDA events. No
 *              memory is allocated.
 * Errors: as fa_fwd_gqa / fa_bwd_gqa for sizes, heads, scale, alignment of
 * the device pointers and the workspace (host pointers have no alignment
 * rule); a NULL struct or a NULL pointer it must hold, or n_chunks < 0 ->
 * FA_ERR_INVALID_ARG. FA_ERR_CUDA when a copy, event or launch fails after
 * part of the work was queued; `stream` is still ordered after whatever was.
 */
int fa_fwd_host(const fa_tensors* host, const fa_tensors* dev, int B, int H, int Hkv, int N, int d,
                float scale, int causal, int n_chunks, void* stream);
int fa_fwd_bwd_host(const fa_tensors* host, const fa_tensors* dev, void* workspace, size_t ws_bytes,
                    int B, int H, int Hkv, int N, int d, float scale, int causal, int n_chunks,
                    void* stream);

/* Size in bytes of the static scratch area behind fa_bwd_noalloc (32 MiB). */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * fa_bwd for callers that cannot allocate device memory. The pages this
 * library follows have no counterpart to this call; it exists for hosts
 * that hand a plug-in no allocator (all device memory belongs to the host's
 * own fixed pool), runtimes that forbid device allocation after start-up,
 * and code that cannot afford cudaMalloc's implicit device-wide
 * synchronisation.
 *
 * Same arguments and results as fa_bwd, minus the workspace: the scratch
 * (the fp32 D vector, fa_bwd_workspace_bytes(B,H,N,d) bytes) is a
 * file-scope __device__ array of FA_BWD_NOALLOC_SCRATCH_BYTES inside
 * the library image, held on every GPU that loads the library until the
 * process exits. The call itself allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine). Its kernels run one after another
 * on `stream`, in the order fa_bwd takes for the same sizes
 * (fa_bwd_fuses_d), so its results equal fa_bwd's bit for bit.
 *   - Problems whose scratch need exceeds FA_BWD_NOALLOC_SCRATCH_BYTES are
 *     rejected with FA_ERR_WORKSPACE before anything is launched
 *     (B*H*N*4 bytes: up to 8,388,608 query rows over all heads).
 *   - Every call looks up the array's device address on the current
 *     device (a runtime query, nothing launched), so the address stays
 *     right after a device reset. The first call on a device may load the
 *     library's device code; make it before any stream capture. Later
 *     calls can be captured into a CUDA graph.
 *   - Every call on a device shares the one array. Calls whose kernels
 *     overlap on the GPU (different streams or host threads without
 *     ordering between them) race on it and give undefined results; order
 *     such calls on one stream. The array keeps the last call's contents;
 *     each call rewrites D before anything reads it.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, void* stream);

/*
 * Row softmax, y_ij = e^(x_ij − m_i) / Σ_j e^(x_ij − m_i) with m_i = max_j
 * x_ij, over x [rows][n] fp32 (row-major, contiguous) into y [rows][n] fp32.
 * y may equal x (in place). Two ways of reaching the same result:
 *   fa_softmax_safe    three passes over each row (maximum; sum of
 *                      e^(x − m); output), the safe softmax of the dcwnkz.com
 *                      GPU-tricks article (appendix on softmax) and of the
 *                      CMU 10-423 L17–L18 notes (section 前置二：online softmax);
 *   fa_softmax_online  two passes: the running maximum and the running
 *                      denominator in one pass, the denominator rescaled by
 *                      e^(m_old − m_new) whenever the maximum grows (same CMU
 *                      section), then the output pass.
 * Exponentials use the hardware 2^x approximation; results match the exact
 * softmax to a few units in the last place of fp32 per element (the sum
 * adds rounding that grows with n). A row of only -inf gives NaN.
 * Errors: null pointer, rows < 1 or n < 1 -> FA_ERR_INVALID_ARG; rows >
 * 2^31 - 1 -> FA_ERR_UNSUPPORTED; x or y not 4-byte aligned ->
 * FA_ERR_MISALIGNED. 16-byte loads are used when n % 4 == 0 and both
 * pointers are 16-byte aligned.
 */
int fa_softmax_safe(const float* x, float* y, long long rows, int n, void* stream);
int fa_softmax_online(const float* x, float* y, long long rows, int n, void* stream);

/*
 * Row softmax from host memory: copies x_host [rows][n] fp32 into x_dev,
 * runs fa_softmax_online (online != 0) or fa_softmax_safe on the device
 * buffers, and copies y_dev into y_host, in n_chunks pipelined slices of
 * consecutive rows (0 = 8; clamped to rows and 64) so that the copies of
 * one slice overlap another's kernel. Results equal the device call's bit
 * for bit. Ordering, resources and page-locking as in fa_fwd_host.
 * Errors: a NULL pointer, rows or n < 1, n_chunks < 0 -> FA_ERR_INVALID_ARG;
 * rows > 2^31 - 1 -> FA_ERR_UNSUPPORTED; x_dev or y_dev not 4-byte aligned
 * -> FA_ERR_MISALIGNED; FA_ERR_CUDA when a copy, event or launch fails
 * after part of the work was queued.
 */
int fa_softmax_host(const float* x_host, float* y_host, float* x_dev, float* y_dev, long long rows, int n,
                    int online, int n_chunks, void* stream);

/*
 * Merge of partial attention results over disjoint key blocks ("07-16 下午"
 * notes, section 长上下文与序列并行: blocks are not normalised separately and
 * added; each block's normaliser and weighted sum are rescaled by
 * e^(m_block − m_global) first). For each row r:
 *     lse_r = ln Σ_s e^(lse_parts[s][r]),
 *     o_r   = Σ_s e^(lse_parts[s][r] − lse_r) · o_parts[s][r][:]
 *   o_parts    [n_parts][rows][d] fp32, each part normalised within its own
 *              keys (o_s = Σ_j e^(x_j − lse_s) v_j over the part's keys);
 *   lse_parts  [n_parts][rows] fp32 natural log; -inf marks a part with no
 *              key (weight 0);
 *   o          [rows][d] bf16 output, lse [rows] fp32 output. A row whose
 *              parts are all -inf gets o = 0, lse = -inf.
 * Errors: null pointer, n_parts or rows < 1 -> FA_ERR_INVALID_ARG; d not 64
 * or 128 -> FA_ERR_UNSUPPORTED; o_parts or o not 16-byte aligned, lse_parts
 * or lse not 4-byte aligned -> FA_ERR_MISALIGNED.
 */
int fa_attn_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse,
                  long long rows, int d, void* stream);

/*
 * Decode step against a paged KV cache. A paged cache (CMU 10-423 notes,
 * section 解碼端：PagedAttention) cuts each request's keys and values into
 * blocks of block_size tokens stored anywhere; a block table maps the
 * request's logical block i to a physical block. In a decode step ("07-16
 * 下午" notes, section Prefill、Decode 与推理调度) each request brings one new
 * token whose query attends to all of that request's cached tokens; the
 * caller has already written the new token's key and value into the cache.
 *   q            [B][H][d] bf16: the new token's query rows.
 *   k_cache,     [num_blocks][Hkv][block_size][d] bf16 each: token t of
 *   v_cache      request b is in block block_table[b][t / block_size], slot
 *                t % block_size (layout chosen here; the pages fix none).
 *   block_table  [B][max_blocks_per_seq] int32 device array.
 *   seq_lens     [B] int32 device array: cached tokens per request (clamped
 *                to [0, max_blocks_per_seq·block_size]; 0 gives o = 0,
 *                lse = -inf).
 *   o, lse       [B][H][d] bf16 and [B][H] fp32 outputs: attention of each
 *                query row over its request's tokens (no mask beyond the
 *                context length); query head h reads K/V head h / (H/Hkv).
 *   workspace    device buffer of fa_decode_workspace_bytes(B, H, d,
 *                n_splits) bytes (16-byte aligned), for the partial results
 *                (required always; not touched when n_splits = 1).
 *   block_size   any size >= 1. Sizes that are a multiple of 8 dividing 128
 *                load each cache block as one TMA box; others are gathered
 *                token by token (fewer bytes per second).
 *   n_splits     the context of every request is cut into n_splits parts of
 *                whole 128-token tiles, processed in parallel and combined
 *                as in fa_attn_merge (two kernels on `stream`). With
 *                n_splits = 1 one kernel writes o and lse directly.
 * Errors: null pointer, sizes < 1, Hkv not dividing H, bad scale ->
 * FA_ERR_INVALID_ARG; d not 64/128, B > 65535, Hkv·ceil(H/Hkv / 16) > 65535,
 * n_splits > 4096, num_blocks·Hkv·block_size >= 2^32 - 1 (token rows of the
 * cache, indexed in 32 bits) -> FA_ERR_UNSUPPORTED; short workspace ->
 * FA_ERR_WORKSPACE; misaligned ->
 * FA_ERR_MISALIGNED. A block-table entry outside [0, num_blocks) is never
 * dereferenced: the tokens it maps are skipped (the results are then
 * undefined) and fa_last_device_error reports FA_ERR_BAD_INDEX.
 */
size_t fa_decode_workspace_bytes(int B, int H, int d, int n_splits);
int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                    const int* seq_lens, void* o, float* lse, void* workspace, size_t ws_bytes, int B,
                    int H, int Hkv, int d, int num_blocks, int block_size, int max_blocks_per_seq,
                    float scale, int n_splits, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word set by
 * any kernel of this library on the current device. Returns FA_OK,
 * FA_ERR_TIMEOUT (a pipeline wait gave up; outputs of the calls since the
 * last check are undefined), FA_ERR_BOUNDS (FA_DEBUG build only: an address
 * a kernel computed fell outside its buffer; that access was skipped and the
 * outputs are undefined), FA_ERR_BAD_INDEX (a decode block table pointed
 * outside the cache) or FA_ERR_CUDA.
 */
int fa_last_device_error(void* stream);

/*
 * Self-test of the device error path. Launches one warp on `stream` that
 * waits on an mbarrier nothing arrives on, through the same bounded wait
 * every kernel of this library uses; the wait gives up after its limit
 * (2 s) and the kernel returns. The next fa_last_device_error then returns
 * FA_ERR_TIMEOUT, and the context stays usable. Reads and writes no caller
 * memory. Returns FA_OK when the launch was enqueued, else FA_ERR_CUDA.
 */
int fa_selftest_wait_limit(void* stream);

/* Human-readable name of an fa_status value (static string). */
const char* fa_status_string(int status);

/* Library version, e.g. "0.1.0". */
const char* fa_version(void);

/*
 * 1 when this library is the FA_DEBUG build (libfa_debug.so), else 0. That
 * build checks every address the kernels compute themselves (all global
 * loads and stores other than TMA tensor copies, the decode kernel's bulk
 * copies, and the shared-memory staging of outputs) against the extent of
 * its buffer; a failed check skips the access and records FA_ERR_BOUNDS for
 * fa_last_device_error. No check traps. It stands in for a memory checker:
 * results on valid inputs equal the release build's bit for bit.
 * Pure host function; needs no GPU.
 */
int fa_debug_checks(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
