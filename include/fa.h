/*
 * fa.h -- C ABI of libfa.so: the FlashAttention-2 forward pass on one GB300
 * (sm_103a), as hand-written CUDA kernels.
 *
 * The operation (sources: "Extend Thunder with CUDA-Python", function
 * flash_attention_reference, and "Blackwell Attention Example", section
 * "Attention Kernel Implementation", blackwell_attention_kernel):
 *
 *   for every batch b < B, head h < H, query row i < N_q:
 *     s_ij      = scale * sum_{c<d} Q[b,h,i,c] * K[b,h,j,c]    (keys j < N_k)
 *     visible j = all j < N_k, or only j <= i when is_causal (top-left
 *                 alignment: query and key rows both counted from 0)
 *     LSE[b,h,i] = log sum_{visible j} exp(s_ij)               (natural log)
 *     O[b,h,i,:] = sum_{visible j} exp(s_ij - LSE[b,h,i]) * V[b,h,j,:]
 *
 * computed tile by tile with an online softmax (running row max m and running
 * sum l, O rescaled when m grows), ending with O/l and LSE = m + log(l).
 * Arithmetic: S and O accumulate in fp32; the softmax numerator P is rounded
 * to the input type before P.V (bf16 inputs) or fed as tf32 (fp32 inputs);
 * O is written in the input type, LSE in fp32.
 *
 * Ownership: the caller allocates Q, K, V, O and LSE in device memory and owns
 * the stream.  A call allocates no device memory and is asynchronous on
 * `stream` (a cudaStream_t; NULL = the legacy default stream).  The library is
 * thread-safe; calls on the same stream run in order.
 *
 * Errors: every entry point returns a status and never aborts the process.
 * Argument errors are found on the host before anything is launched.  A
 * device-side pipeline wait that exceeds its time limit (a bounded wait, never
 * a hang) makes the kernel stop, raise a device error word and exit cleanly;
 * fa_check() reports it as FA_ERR_TIMEOUT.  The text of the last error of the
 * calling thread is available from fa_last_error().
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, stride[3] != 1, non-finite scale */
  FA_ERR_UNSUPPORTED = 2,  /* valid arguments the library has no kernel for (head dim, alignment) */
  FA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed (launch, attribute, device query) */
  FA_ERR_TIMEOUT = 4       /* a kernel's bounded pipeline wait expired; its outputs are undefined */
} fa_status_t;

typedef enum {
  FA_BF16 = 0,  /* Q, K, V, O bf16; tensor-core kind::f16 */
  FA_FP32 = 1   /* Q, K, V, O fp32; tensor-core kind::tf32 (d = 64, 128) or CUDA-core fp32 (d = 16, 32) */
} fa_dtype_t;

/* A [B, H, N, d] view: element [b,h,n,c] lives at
 * ptr + (b*stride[0] + h*stride[1] + n*stride[2] + c*stride[3]) elements.
 * stride[3] must be 1 (each row of d values is contiguous). */
typedef struct {
  void* ptr;
  int64_t stride[4];
} fa_tensor_t;

/*
 * fa_fwd -- O, LSE = attention(Q, K, V, scale, is_causal).
 *
 *   dtype          element type of Q, K, V and O (LSE is always fp32).
 *   B, H           batch and head counts (>= 1); Q, K, V, O share them.
 *   N_q, N_k       query and key/value sequence lengths (>= 1).
 *   d              head dimension of Q, K, V and O (the same for V).
 *   Q              [B, H, N_q, d] device view.
 *   K, V           [B, H, N_k, d] device views.
 *   scale          multiplier of Q.K (finite; 1/sqrt(d) is the usual choice).
 *   is_causal      0: no mask; 1: top-left causal mask (key j visible to
 *                  query row i iff j <= i); 2: bottom-right alignment (j <=
 *                  i + N_k - N_q; with N_q > N_k the first rows see no key and
 *                  get O = 0, LSE = -inf).
 *   O              [B, H, N_q, d] device view, written.  Must not overlap the inputs.
 *   LSE            fp32 [B, H, N_q] device array written at
 *                  LSE + b*lse_stride[0] + h*lse_stride[1] + i*lse_stride[2],
 *                  or NULL to skip it (lse_stride is then ignored).
 *   stream         cudaStream_t to launch on.
 *
 * Supported: d in {16, 32} on the small-head path (any alignment); any other
 * d that makes a row a multiple of 16 bytes (d % 8 == 0 in bf16, d % 4 == 0
 * in fp32), up to 256 in bf16 and 128 in fp32, on the tensor-core path, which
 * also needs 16-byte aligned Q/K/V/O base pointers and strides[0..2] * element
 * size that are multiples of 16 bytes (FA_ERR_UNSUPPORTED otherwise).  The
 * tensor-core tiles have 64, 128 or (bf16, head dims above 128) 256 columns: a
 * smaller d is computed on tiles whose extra columns are loaded as zeros
 * (exact: they add nothing to Q.K and give O columns that are not stored), so
 * d = 96 costs the tensor work of d = 128.  Any N_q, N_k >= 1: the tail of a
 * tile is masked, not required to divide.
 */
fa_status_t fa_fwd(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k,
                   int64_t d, const fa_tensor_t* Q, const fa_tensor_t* K,
                   const fa_tensor_t* V, float scale, int is_causal,
                   const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                   void* stream);

/*
 * fa_fwd_gqa -- fa_fwd with grouped K/V heads (grouped-query attention): K and
 * V are [B, H_kv, N_k, d] and query head h attends to K/V head h / (H / H_kv).
 * H_kv must divide H (FA_ERR_INVALID_ARG otherwise); H_kv = H is fa_fwd.
 * Other arguments and rules as fa_fwd.
 */
fa_status_t fa_fwd_gqa(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k,
                       int64_t d, const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                       int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3], void* stream);

/*
 * fa_fwd_ws -- fa_fwd_gqa with a caller-owned workspace, which the fp32
 * tensor-core path uses to hold V transposed ("Blackwell Attention Example",
 * section "Attention Kernel Implementation": O accumulates P.V tile by tile).
 *
 * Why: with fp32 inputs both contractions run on the tf32 tensor cores, which
 * take their operands only with the reduction index contiguous; for P.V that
 * index is the key, and V [B, H_kv, N_k, d] has the head dims contiguous.
 * fa_fwd transposes every V tile in shared memory, once per query tile that
 * reads it.  fa_fwd_ws first writes V^T once into `workspace` (one pass that
 * reads and writes V's bytes), and the attention kernel then loads V^T tiles
 * the way it loads K tiles -- faster whenever a V tile is read by two or more
 * query tiles.  The results equal fa_fwd's up to the order of fp32 additions.
 *
 *   workspace        device memory of at least fa_fwd_ws_bytes(dtype, B, H,
 *                    H_kv, N_q, N_k, d) bytes, 256-byte aligned, owned by the
 *                    caller; its contents are scratch (V^T, fp32
 *                    [B * H_kv][d][N_k rounded up to 32]).  Calls that may
 *                    overlap on the device need separate workspaces.
 *   workspace_bytes  its size; less than required is FA_ERR_INVALID_ARG.
 *   other arguments  as fa_fwd_gqa.
 *
 * fa_fwd_ws_bytes is 0 where no workspace is used: bf16 inputs, the
 * small-head path (d = 16, 32), and fp32 problems whose V tiles are each read
 * by a single query tile (ceil(N_q / 128) * H / H_kv == 1); fa_fwd_ws is then
 * fa_fwd_gqa and `workspace` may be NULL.  It is also 0 for arguments that
 * fa_fwd_gqa rejects.
 */
size_t fa_fwd_ws_bytes(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d);

fa_status_t fa_fwd_ws(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                      const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                      int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                      void* workspace, size_t workspace_bytes, void* stream);

/* One problem of a grouped call: the arguments of fa_fwd_gqa, by value.
 * H_kv = 0 means H_kv = H (K and V have the query heads).
 * Dv: head dim of V and O when it differs from d ("Blackwell Attention
 * Example", blackwell_attention: Q and K share d, V and O have Dv columns);
 * 0 means Dv = d.  V is then [B, H_kv, N_k, Dv] and O [B, H, N_q, Dv].  A
 * problem with Dv != d takes the tensor-core path (Dv up to 256 in bf16, 128
 * in fp32, a multiple of 16 bytes like d); fa_fwd_grouped with one problem is
 * the entry point for it. */
typedef struct {
  int64_t B, H, N_q, N_k, d;
  fa_tensor_t Q, K, V, O;
  float* LSE;
  int64_t lse_stride[3];
  float scale;
  int is_causal;
  int64_t H_kv;
  int64_t Dv;
} fa_problem_t;

/*
 * fa_fwd_grouped -- several independent problems of one dtype.
 *
 * Problems that take the small-head path (d in {16, 32}) all run in ONE
 * launch; this is how the row and the column attention of the axial workload
 * (both strided views of the same [B, H, W, heads, hd] tensors) are computed
 * together.  Any other problem is launched on its own, in order, on `stream`.
 * Validation of every problem happens before any launch; n = 0 is a no-op.
 */
fa_status_t fa_fwd_grouped(fa_dtype_t dtype, int n, const fa_problem_t* problems, void* stream);

/*
 * Split-KV forward: the same operation as fa_fwd, with the key range of every
 * 256-row query tile cut into n_split balanced parts that run as separate
 * work units.  It serves problems with few query tiles for the number of SMs
 * (long keys, short queries): more units fill the last wave of the persistent
 * grid.  Each unit writes its normalised partial output O_s (fp32) and its
 * log-sum-exp L_s into `workspace`; a second kernel merges them with
 * L = log sum_s e^{L_s} and O = sum_s e^{L_s - L} O_s (the rescaling identity
 * of the online softmax in "Extend Thunder with CUDA-Python",
 * flash_attention_reference).
 *
 *   n_split          1..8; 1 is exactly fa_fwd (workspace unused).  Non-causal
 *                    and causal problems alike; a tile with fewer key tiles
 *                    than n_split uses fewer parts.
 *   workspace        device memory of at least
 *                    fa_fwd_splitkv_workspace_bytes(B, H, N_q, d, n_split)
 *                    bytes, 256-byte aligned, owned by the caller; its
 *                    contents are scratch.  Concurrent calls need separate
 *                    workspaces.
 *   other arguments  as fa_fwd; only the tensor-core path (d = 64, 128)
 *                    splits (FA_ERR_UNSUPPORTED otherwise).
 */
size_t fa_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t N_q, int64_t d, int n_split);

/* Split count for this problem on the current device (1 = do not split).
 * It models the run as waves of one work unit per SM and takes a split only
 * when that model is at least 10 % faster and every part keeps >= 1024 keys.
 * Causal problems (their longest-first schedule already balances them) and
 * FA_FP32 problems (splitting was slower on the shapes measured) return 1;
 * fa_fwd_splitkv still accepts an explicit n_split for them.  Errors (no
 * device, bad sizes) also return 1. */
int fa_fwd_splitkv_choose(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                          int is_causal);

fa_status_t fa_fwd_splitkv(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                           const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                           int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                           int n_split, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory.  The source pages have no counterpart to this entry point:
 * it exists only for how a caller manages memory, not for what is computed.
 *
 * Who needs it: a caller with no device allocator of its own (a plain C
 * host program that does not want to own and size a workspace), and a caller
 * that must not call cudaMalloc / cudaFree on its hot path, because those
 * calls can synchronise the device, take driver locks, or fail with
 * out-of-memory at a point where the caller cannot recover (a latency-bound
 * serving loop, a real-time thread).  This call allocates nothing: the
 * partial results go to one fixed scratch buffer per device that is part of
 * the library image, FA_SPLITKV_NOALLOC_SCRATCH_BYTES (128 MiB) in size.
 *
 *   Arguments   as fa_fwd_splitkv, without the workspace.  n_split = 1 is
 *               fa_fwd and uses no scratch; fa_fwd_splitkv_choose gives a
 *               good n_split.
 *   Size limit  a problem whose scratch need,
 *               fa_fwd_splitkv_workspace_bytes(B, H, N_q, d, n_split), is
 *               above FA_SPLITKV_NOALLOC_SCRATCH_BYTES is rejected on the
 *               host with FA_ERR_UNSUPPORTED and a message giving both sizes
 *               (nothing is launched): use fewer splits, or fa_fwd_splitkv
 *               with your own workspace.
 *   First call  on each device, the first call (with that device current)
 *               looks up the scratch buffer's device address; that lookup
 *               makes the CUDA runtime load this part of the library onto
 *               the device.  Make that first call before any stream capture
 *               on the device.
 *   Races       there is ONE buffer per device.  Calls that can overlap on
 *               the device (different streams, or different host threads
 *               without ordering between their streams) race on it and give
 *               wrong results.  Calls issued in order on one stream are safe.
 *   Contents    every scratch element the merge step reads is first written
 *               by the same call, so nothing needs clearing between calls.
 *   Residency   the buffer is part of the library's device image.  Under
 *               lazy module loading (the CUDA default) a device holds it
 *               from the first call on that device until the process exits;
 *               under eager loading (CUDA_MODULE_LOADING=EAGER) every device
 *               on which the process creates a context holds it from then
 *               on, whether or not this entry point is ever called.
 *   Device reset  the buffer's address is looked up once per device and kept
 *               (as is the library's error word): calling cudaDeviceReset
 *               while this library is loaded is not supported.
 */
#define FA_SPLITKV_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20)

fa_status_t fa_fwd_splitkv_noalloc(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                                   const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                                   int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                                   int n_split, void* stream);

/*
 * fa_bwd -- backward of fa_fwd: dQ, dK, dV of sum(dO * O) ("Blackwell
 * Attention Example", section "Backward Kernel Implementation": the row-sum
 * preprocess delta = rowsum(dO * O) and the products dV = P^T dO,
 * dS = P * (dO V^T - delta), dQ = scale * dS K, dK = scale * dS^T Q, with
 * P recomputed from Q, K and the forward's LSE).
 *
 *   dtype          FA_BF16 (FA_ERR_UNSUPPORTED for FA_FP32); every tensor bf16.
 *   d              a multiple of 8 up to 128 (64 and 128 fill the kernel's
 *                  tiles; other head dims run on 64- or 128-column tiles
 *                  whose extra columns load as zeros).
 *   Q, K, V        the forward's inputs; O and LSE / lse_stride its outputs
 *                  (LSE natural log, as fa_fwd writes it).  Same views and
 *                  rules as fa_fwd (16-byte aligned bases and strides).
 *   dO             incoming gradient, [B, H, N_q, d] like O.
 *   dQ, dK, dV     outputs, shaped like Q, K, V (any strides meeting the same
 *                  alignment rules); every element is written.  Keys that no
 *                  query sees (causal, N_k > N_q) get zero gradients.
 *   scale, is_causal  as in the forward call.
 *   workspace      device memory of at least fa_bwd_workspace_bytes(B, H,
 *                  N_q, d) bytes (fa_bwd_dv: N_q, max(d, d_v)), 256-byte
 *                  aligned, caller-owned scratch (an fp32 dQ accumulator of the
 *                  tile's width and two per-row vectors).  Concurrent calls need
 *                  separate workspaces.
 * Asynchronous on `stream` (three kernels).  Argument errors are reported on
 * the host before any launch.
 */
size_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N_q, int64_t d);

/*
 * fa_bwd_gqa -- fa_bwd with grouped K/V heads: K, V, dK and dV are
 * [B, H_kv, N_k, d], H_kv divides H, and dK, dV of a K/V head sum the
 * gradients of the H / H_kv query heads that read it.  The workspace size is
 * fa_bwd_workspace_bytes(B, H, N_q, d) (query heads).  Other arguments as
 * fa_bwd.
 */
/*
 * fa_bwd_dv -- fa_bwd_gqa with V, O, dO and dV of head dim d_v ("Blackwell
 * Attention Example", blackwell_attention takes V with Dv columns): Q, K, dQ,
 * dK are [.., d], V, dV [B, H_kv, N_k, d_v], O, dO [B, H, N_q, d_v]; d and d_v
 * multiples of 8 up to 128.  Workspace: fa_bwd_workspace_bytes(B, H, N_q,
 * max(d, d_v)).  Other arguments as fa_bwd_gqa.
 */
fa_status_t fa_bwd_dv(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                      int64_t d_v, const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V,
                      const fa_tensor_t* O, const fa_tensor_t* dO, const float* LSE, const int64_t lse_stride[3],
                      float scale, int is_causal, const fa_tensor_t* dQ, const fa_tensor_t* dK,
                      const fa_tensor_t* dV, void* workspace, size_t workspace_bytes, void* stream);

fa_status_t fa_bwd_gqa(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                       const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, const fa_tensor_t* O,
                       const fa_tensor_t* dO, const float* LSE, const int64_t lse_stride[3], float scale,
                       int is_causal, const fa_tensor_t* dQ, const fa_tensor_t* dK, const fa_tensor_t* dV,
                       void* workspace, size_t workspace_bytes, void* stream);

fa_status_t fa_bwd(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                   const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, const fa_tensor_t* O,
                   const fa_tensor_t* dO, const float* LSE, const int64_t lse_stride[3], float scale, int is_causal,
                   const fa_tensor_t* dQ, const fa_tensor_t* dK, const fa_tensor_t* dV, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * fa_fwd_varlen -- fa_fwd_gqa over B packed sequences of different lengths
 * (variable-length batch): sequence b has queries at packed rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and keys at cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1, and attends only within itself.
 *
 *   cu_seqlens_q, cu_seqlens_k  device int32 arrays of B + 1 non-decreasing
 *                  offsets starting at 0, ending at total_q / total_k.  They
 *                  are read on the device: not validated on the host (a row
 *                  whose packed index falls outside [0, total_q) is not
 *                  written).  Sequences may be empty.
 *   total_q, total_k  packed rows (>= 1 each); max_len_q  host upper bound of
 *                  the query lengths, 1 .. total_q (it sizes the tile grid:
 *                  query rows of a sequence past max_len_q are not computed).
 *   d, d_v         head dims of Q, K and of V, O (d_v = 0 means d_v = d).
 *   Q              [1, H, total_q, d] view (stride[1] head, stride[2] row),
 *                  K [1, H_kv, total_k, d], V [1, H_kv, total_k, d_v],
 *                  O [1, H, total_q, d_v]; the rules of fa_fwd.
 *   LSE            [1, H, total_q] (lse_stride[1] head, [2] row), or NULL.
 *   is_causal      0, 1 (top-left) or 2 (bottom-right), per sequence.
 * Supported: bf16, d and d_v multiples of 8 up to 128, always on the
 * tensor-core path (FA_ERR_UNSUPPORTED otherwise).
 */
fa_status_t fa_fwd_varlen(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t total_q, int64_t total_k,
                          int64_t max_len_q, int64_t d, int64_t d_v, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k,
                          const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                          int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                          void* stream);

/*
 * fa_axial_block_fwd -- the axial attention block of the axial-attention
 * transcript (its module's forward), fused per sequence, fp32: on x
 * [B, H, W, D] (contiguous), a row pass over the W-long rows and then a
 * column pass over the H-long columns of the updated grid, each
 *     x += out_proj(attention(qkv_proj(LayerNorm(x))))
 * with LayerNorm (biased variance, eps 1e-5, weight and bias), a bias-free
 * QKV projection (qkv_w [3D, D], rows q | k | v, as nn.Linear's weight),
 * softmax(q k^T / sqrt(D / heads)) v per head and an output projection
 * (out_w [D, D], out_b [D]).
 *
 *   Supported: D = 64, heads = 4, 1 <= H, W <= 32 (FA_ERR_UNSUPPORTED
 *   otherwise); x, out and every weight 16-byte aligned.
 *   out            [B, H, W, D], written; may be x (in place).
 * Asynchronous on `stream` (two launches).
 */
typedef struct {
  const float* norm_w; /* [D] */
  const float* norm_b; /* [D] */
  const float* qkv_w;  /* [3D, D] */
  const float* out_w;  /* [D, D] */
  const float* out_b;  /* [D] */
} fa_axial_weights_t;

fa_status_t fa_axial_block_fwd(int64_t B, int64_t H, int64_t W, int64_t D, int64_t heads, const float* x,
                               const fa_axial_weights_t* row, const fa_axial_weights_t* col, float* out,
                               void* stream);

/*
 * fa_check -- synchronise `stream`, then read and clear the device error word
 * raised by kernels launched from this library on the current device.
 * Returns FA_OK, FA_ERR_TIMEOUT (a bounded wait expired in some launch since
 * the last check) or FA_ERR_CUDA (the stream reported an error).
 */
fa_status_t fa_check(void* stream);

/* Static description of a status code. */
const char* fa_status_string(fa_status_t status);

/* Detail of the last non-OK status returned to the calling thread ("" if none). */
const char* fa_last_error(void);

/*
 * Test hooks (process-wide; not for production use).
 *   timeout_ns   limit of every device-side pipeline wait (0 = default, 1 s).
 *   debug_flags  bit 0: the load warp of the forward kernels withholds one K
 *                tile (the second of work unit 0) and the backward's one
 *                Q/dO step of block 0, so the consumer's bounded wait runs
 *                out and the launch ends with FA_ERR_TIMEOUT instead of a hang.
 */
void fa_debug_set(uint64_t timeout_ns, int debug_flags);

/* ABI version of this header (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
