/*
 * fa2.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 forward library
 * (libfa2_gb300.so).
 *
 * The operation ("From FlashAttention to FlashAttention 2", FlashAttention 2:
 * What Changed and Layer 5: The Forward Kernel; "FlashAttention-2 from PyTorch
 * to Triton", introduction and the Triton kernel; "Writing FlashAttention 2 in
 * Triton", Steps 1-6): for every batch b, head h and query row i,
 *     O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j) v_j
 *     L[b,h,i]   = log sum_j exp(scale * q_i . k_j)        (natural log)
 * over the visible keys j: j < N, and j <= i when causal (top-left aligned,
 * "Writing FlashAttention 2 in Triton", Step 4).  The library computes it tile by
 * tile with the online-softmax recurrence and never forms the N x N scores.
 *
 * Conventions for every entry point:
 *   - Pointers named q, k, v, o, lse are DEVICE pointers on the current CUDA
 *     device, owned by the caller, which allocates and frees them.  The library
 *     allocates no device memory, keeps no pointer after the call returns and
 *     never synchronises the stream.
 *   - Layouts are contiguous row-major: q and o are [B, H, M, D], k and v are
 *     [B, H, N, D] (the problem statement of the pages: Q [B,H,M,D], K/V
 *     [B,H,N,D], O [B,H,M,D]); lse is [B, H, M] fp32.  Element type of q, k, v, o
 *     is `dtype`: FA2_BF16 (bfloat16) or FA2_FP32 (fp32 storage; the products run
 *     on the tensor cores as TF32 with fp32 accumulation).
 *   - q, k, v and o must be 16-byte aligned (TMA); lse 4-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  A return of FA2_OK means the kernel was launched; results are
 *     valid once the stream has reached that point.
 *   - Errors are returned as negative status codes; nothing is launched on
 *     error.  No exception crosses the ABI and the library never exits the
 *     process.  fa2_strerror() names each code.
 *   - The first call on a device sets up per-device state that later calls
 *     reuse (the device address of the status word, the host-buffer entries'
 *     copy streams, the built-in buffer of fa2_fwd_splitkv_noalloc).  It belongs
 *     to the device's primary context: after a cudaDeviceReset of that device the
 *     state is stale, and the library must not be used on it again in the same
 *     process.
 */
#ifndef FA2_GB300_H
#define FA2_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of q, k, v and o. */
#define FA2_BF16 0
#define FA2_FP32 1

/* Status codes. */
#define FA2_OK 0
#define FA2_ERR_NULL (-1)           /* a required pointer is NULL */
#define FA2_ERR_SHAPE (-2)          /* B, H, M or N <= 0, or H_kv <= 0 or not dividing H */
#define FA2_ERR_HEADDIM (-3)        /* D is not 64 or 128 */
#define FA2_ERR_DTYPE (-4)          /* dtype is not FA2_BF16 or FA2_FP32 */
#define FA2_ERR_ALIGN (-5)          /* q/k/v/o not 16-byte or lse not 4-byte aligned */
#define FA2_ERR_SCALE (-6)          /* scale is not finite and > 0 */
#define FA2_ERR_TOO_LARGE (-7)      /* sizes exceed the grid or tensor-map limits */
#define FA2_ERR_ARCH (-8)           /* current device is not compute capability 10.3 */
#define FA2_ERR_CUDA (-9)           /* a CUDA runtime or driver call failed */
#define FA2_ERR_DEVICE_TIMEOUT (-10) /* a kernel gave up on a pipeline wait (see fa2_device_status) */
#define FA2_ERR_WORKSPACE (-11)     /* workspace missing, misaligned or too small */
#define FA2_ERR_MODIFIER (-12)      /* softcap < 0 or not finite, or alibi_batch_stride not 0 or H */

/*
 * fa2_fwd -- FlashAttention-2 forward pass.
 *
 * Computes O and L as defined above for all B*H heads.
 *   q      [B,H,M,D] queries            k, v  [B,H,N,D] keys and values
 *   o      [B,H,M,D] output (written)   lse   [B,H,M] fp32 logsumexp (written)
 *   B, H   batch size and number of heads (> 0)
 *   M, N   query and key sequence lengths (> 0, any value: ragged tails are
 *          masked, "FlashAttention-2 from PyTorch to Triton", the ragged-tile fix)
 *   D      head dimension: 64 or 128
 *   scale  softmax scale applied to q.k, finite and > 0 (usually 1/sqrt(D))
 *   causal 0: every key visible; nonzero: key j visible to query i iff j <= i
 *   dtype  FA2_BF16 or FA2_FP32
 *   stream cudaStream_t to launch on
 * Returns FA2_OK or a negative FA2_ERR_* code.  Inputs are only read; o and lse
 * are fully overwritten (rows i < M only; memory past the tensors is untouched).
 */
int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
            int M, int N, int D, float scale, int causal, int dtype, void* stream);

/*
 * fa2_fwd_gqa -- the same forward pass with grouped-query (or multi-query)
 * attention: k and v hold H_kv heads, [B, H_kv, N, D], H_kv divides H, and query
 * head h attends to key/value head h / (H / H_kv) of the same batch entry
 * ("From FlashAttention to FlashAttention 2", Layer 8: Multi-Query / Grouped-Query
 * Attention).  H_kv == H is fa2_fwd; H_kv == 1 is multi-query attention.  All
 * other arguments, layouts, ownership and errors are those of fa2_fwd.
 */
int fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int H_kv, int M, int N, int D, float scale, int causal, int dtype, void* stream);

/*
 * Split-KV forward ("From FlashAttention to FlashAttention 2", Layer 2: the
 * split-KV dispatch when num_splits > 1).  When B*H*(query tiles) cannot fill the
 * GPU (short M, long N), the key range is cut into num_splits slices: each slice
 * computes a partial result over its keys (O_s normalised by its own row sum,
 * L_s = its logsumexp) into `workspace`, and a combine kernel merges them into O
 * and L:  L = ln sum_s exp(L_s),  O = sum_s exp(L_s - L) O_s.  The result is the
 * same attention as fa2_fwd_gqa (up to rounding).
 *
 *   num_splits  number of key slices; <= 0 picks fa2_splitkv_num_splits(); it is
 *               reduced so that no slice is empty (at most ceil(N/128) slices)
 *               and capped at 64; 1 runs the plain forward (workspace unused)
 *   workspace   caller-owned DEVICE buffer, 256-byte aligned, of at least
 *               fa2_splitkv_workspace_bytes(B, H, M, D, num_splits) bytes; its
 *               contents on entry are ignored and on return are scratch
 * All other arguments as fa2_fwd_gqa.  Returns FA2_ERR_WORKSPACE if the workspace
 * is needed and missing, misaligned or too small.  Two kernels are launched on
 * `stream`; concurrent calls must not share a workspace.
 */
int fa2_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int H_kv, int M, int N, int D, float scale, int causal, int dtype,
                    int num_splits, void* workspace, size_t workspace_size, void* stream);

/* Split count fa2_fwd_splitkv uses when given num_splits <= 0, for the current
 * device (about one wave of CTAs, at least 4 key tiles per slice; H_kv counts
 * because a CTA serves two query heads of a group when M <= 128); >= 1, or a
 * negative FA2_ERR_* code for invalid sizes or when the device cannot be queried. */
int fa2_splitkv_num_splits(int B, int H, int H_kv, int M, int N, int D, int dtype);

/* Workspace bytes fa2_fwd_splitkv needs for num_splits slices (0 if num_splits <= 1
 * or the sizes are invalid): num_splits * B*H*M * (D + 1) * 4 plus padding. */
size_t fa2_splitkv_workspace_bytes(int B, int H, int M, int D, int num_splits);

/*
 * fa2_fwd_splitkv_noalloc -- fa2_fwd_splitkv for callers that cannot allocate
 * device memory (an exhausted or locked-down allocator, a host framework that
 * owns every allocation, or code that must not call cudaMalloc/cudaFree because
 * they synchronise the device).  The split-KV partials go to a buffer built into
 * the library: a 32 MiB array in device memory that every GPU which loads the
 * library's device code holds until the process exits.  This call allocates
 * nothing.  The pages have no counterpart to it; it is an interface addition.
 *
 * Arguments as fa2_fwd_splitkv, without the workspace.  Limit: the partials of
 * the split actually run (num_splits after fa2_fwd_splitkv lowers it: the
 * automatic choice for <= 0, at most 64 and at most ceil(N/128) slices) take
 * fa2_splitkv_workspace_bytes(B, H, M, D, that count) bytes and must fit in the
 * 32 MiB buffer, else FA2_ERR_WORKSPACE is returned and nothing runs (pass a
 * smaller num_splits, or use fa2_fwd_splitkv with your own workspace).
 * The first call on a device, with that device current, looks up the buffer's
 * device address (and may load the library's device code); make that first call
 * before any stream capture.  The address is cached for the device's primary
 * context: after a cudaDeviceReset the library's per-device state, this address
 * included, is stale and the library must not be used on that device again in
 * the same process.  All calls on a device share the one buffer, which keeps the
 * previous call's contents (nothing in it needs to start at zero): calls whose
 * kernels may overlap on the GPU (different streams without ordering, or several
 * threads) race on it and must be serialised by the caller.
 */
int fa2_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int H_kv, int M, int N, int D, float scale, int causal,
                            int dtype, int num_splits, void* stream);

/*
 * fa2_fwd_ext -- the forward pass with score modifiers: a sliding window, a
 * softcap and ALiBi biases ("From FlashAttention to FlashAttention 2", Layer 1:
 * Python API, the window_size, softcap and alibi_slopes options; "Writing
 * FlashAttention 2 in Triton", What to do after your FA2 works: the sliding-window
 * mask as a change of the causal mask formula, ALiBi as a bias added to the
 * score).  For query row i of head (b, h) and key j:
 *     s = scale * q_i . k_j
 *     s = softcap * tanh(s / softcap)                     when softcap > 0
 *     s = s - alibi_slopes[b * alibi_batch_stride + h] * |i - j|
 *                                                         when alibi_slopes != NULL
 * and key j is visible iff j < N, j >= i - window_left (when window_left >= 0),
 * j <= i + window_right (when window_right >= 0) and j <= i (when causal).  O and
 * L are the softmax-weighted sum and the logsumexp of s over the visible keys; a
 * row with no visible key (possible with a window) gets O = 0 and L = -inf.
 *
 *   window_left, window_right  keys before / after the diagonal a row may see;
 *                      negative = unbounded (-1, -1: no window)
 *   softcap            0 = off; otherwise finite and > 0
 *   alibi_slopes       NULL = no ALiBi, or a DEVICE fp32 array (4-byte aligned,
 *                      caller-owned, only read) of H slopes shared by every batch
 *                      entry (alibi_batch_stride 0) or B*H slopes (stride H)
 *   num_splits, workspace, workspace_size   as fa2_fwd_splitkv: 1 = no key
 *                      split (workspace unused), <= 0 = the library's choice
 * Other arguments, layouts and errors as fa2_fwd_gqa, plus FA2_ERR_MODIFIER for an
 * invalid softcap or stride, FA2_ERR_ALIGN for misaligned slopes and
 * FA2_ERR_TOO_LARGE when a modifier is in use and M or N exceeds 2^30.  With no
 * modifier in use this is fa2_fwd_splitkv.
 */
int fa2_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int H_kv, int M, int N, int D, float scale, int causal, int window_left,
                int window_right, float softcap, const float* alibi_slopes,
                int alibi_batch_stride, int dtype, int num_splits, void* workspace,
                size_t workspace_size, void* stream);

/*
 * fa2_bwd -- FlashAttention-2 backward pass ("From FlashAttention to
 * FlashAttention 2", Backward Pass: Recomputation and Layer 7: The Backward
 * Kernel; "FlashAttention-2 from PyTorch to Triton", Known gaps item 5).  Given
 * the forward's inputs, its output o and logsumexp lse, and the upstream
 * gradient dout = dloss/dO, writes
 *     dq = dloss/dq,   dk = dloss/dk,   dv = dloss/dv
 * recomputing P = exp(scale q.k - L) tile by tile:  D_i = rowsum(dout o o),
 * dS = P (dout v^T - D),  dv = P^T dout,  dk = scale dS^T q,  dq = scale dS k.
 * With grouped-query attention dk and dv of a key/value head sum over the query
 * heads that read it.  The pages form dq "by atomics or by a second pass"; this
 * entry takes the first way at D = 128: the dk/dv kernel also forms each step's
 * dS k and adds it into an fp32 accumulator in the workspace with reductions at
 * L2, then a small kernel scales it and rounds it to bf16.  The order of those
 * adds varies between runs, so dq may differ in its last bits from run to run
 * (dk and dv do not).  At D = 64, and in fa2_bwd_deterministic, dq comes from a
 * second pass over the keys instead, and every output is bitwise reproducible.
 *
 *   q, o, dout, dq  [B,H,M,D] bf16          k, v, dk, dv  [B,H_kv,N,D] bf16
 *   lse             [B,H,M] fp32, as written by the forward for the same inputs
 *   causal, scale   as given to the forward
 *   dtype           FA2_BF16 (the only type of this entry; else FA2_ERR_DTYPE)
 *   workspace       caller-owned DEVICE buffer, 256-byte aligned, of at least
 *                   fa2_bwd_workspace_bytes(B, H, M) bytes; scratch on return
 * Device pointers, 16-byte aligned (lse 4-byte); dq, dk, dv are fully
 * overwritten, everything else is only read.  Three kernels (dq by reduction)
 * or four (second pass) are launched on `stream`; concurrent calls must not
 * share a workspace.  Errors as fa2_fwd_gqa, plus FA2_ERR_WORKSPACE and
 * FA2_ERR_TOO_LARGE for M or N above 2^30.
 */
int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
            const void* dout, void* dq, void* dk, void* dv, int B, int H, int H_kv, int M, int N,
            int D, float scale, int causal, int dtype, void* workspace, size_t workspace_size,
            void* stream);

/*
 * fa2_bwd_deterministic -- fa2_bwd with dq always from the second pass over the
 * keys (the pages' alternative to atomics) at both head dims: dq, dk and dv are
 * bitwise reproducible.  Same arguments, workspace and errors as fa2_bwd.
 */
int fa2_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, int B, int H, int H_kv, int M,
                          int N, int D, float scale, int causal, int dtype, void* workspace,
                          size_t workspace_size, void* stream);

/* Workspace bytes fa2_bwd and fa2_bwd_deterministic need: (2 + 128) * B*H * (M
 * rounded up to 128) * 4 -- two fp32 vectors per query row and the fp32 dq
 * accumulator of dq by reduction (0 for invalid sizes). */
size_t fa2_bwd_workspace_bytes(int B, int H, int M);

/*
 * fa2_fwd_host -- the forward for inputs and outputs in HOST memory.  Copies q,
 * k, v from host to the caller's device buffers, runs the forward and copies o
 * and lse back, cut into `chunks` slices of heads (each slice: whole key/value
 * heads with the query heads that read them) so that the copy of one slice
 * overlaps the compute of the previous one and the copy back of the one before.
 * Copies to the device run on a library stream, the kernels on `stream`, copies
 * back on a second library stream; `stream` reaches its next work only after the
 * last copy back, so synchronising `stream` makes o_host and lse_host valid.
 *
 *   q_host, k_host, v_host  [B,H,M,D] / [B,H_kv,N,D] inputs in host memory, only read
 *   o_host, lse_host        [B,H,M,D] / [B,H,M] fp32 outputs in host memory, overwritten
 *   q, k, v, o, lse         DEVICE buffers of the same shapes (caller-owned, as
 *                           fa2_fwd_gqa); q, k, v are overwritten by the copies
 *   chunks                  slices (<= 0: 4); at most B*H_kv and 32
 * Host buffers should be page-locked (cudaHostAlloc or cudaHostRegister): the
 * copies from pageable memory do not overlap anything.  Other arguments and
 * errors as fa2_fwd_gqa.  The library's two copy streams and their events are
 * created on the first call on a device (not during stream capture); calls on
 * one device are enqueued one at a time.  The pages have no counterpart to this
 * entry: it is the host-side pipelining of the same forward.
 */
int fa2_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                 float* lse_host, void* q, void* k, void* v, void* o, float* lse, int B, int H,
                 int H_kv, int M, int N, int D, float scale, int causal, int dtype, int chunks,
                 void* stream);

/*
 * fa2_bwd_host -- the backward for inputs and outputs in HOST memory, pipelined
 * like fa2_fwd_host: slice by slice of whole key/value heads (with the query
 * heads that read them), q, k, v, o, lse and dout are copied in on a library
 * stream, fa2_bwd runs on `stream`, and dq, dk, dv are copied back on a second
 * library stream, so one slice's copies overlap the other slices' kernels.
 * `stream` reaches its next work only after the last copy back.
 *
 *   *_host          host buffers of the fa2_bwd shapes: q, k, v, o, lse, dout are
 *                   only read; dq, dk, dv are overwritten
 *   q ... dv        DEVICE buffers of the same shapes (caller-owned); q, k, v, o,
 *                   lse, dout are overwritten by the copies
 *   workspace       as fa2_bwd, sized for the whole problem (every slice reuses it)
 *   chunks          slices (<= 0: 8 while each slice keeps at least 1.5 waves of
 *                   the dK/dV kernel's CTAs, B*H_kv*ceil(N/128)/8 >= 1.5 * SMs,
 *                   else 4); at most B*H_kv and 32
 * Host buffers should be page-locked.  Other arguments and errors as fa2_bwd and
 * fa2_fwd_host; each slice is its own problem with fa2_bwd's kernels, so dk and
 * dv equal fa2_bwd's bitwise and dq (by reduction at D = 128) within its rounding.
 * The pages have no counterpart to this entry.
 */
int fa2_bwd_host(const void* q_host, const void* k_host, const void* v_host, const void* o_host,
                 const float* lse_host, const void* dout_host, void* dq_host, void* dk_host, void* dv_host,
                 void* q, void* k, void* v, void* o, float* lse, void* dout, void* dq, void* dk, void* dv,
                 int B, int H, int H_kv, int M, int N, int D, float scale, int causal, int dtype,
                 void* workspace, size_t workspace_size, int chunks, void* stream);

/* Static, human-readable name of a status code (never NULL). */
const char* fa2_strerror(int status);

/*
 * fa2_device_status -- read the sticky device-side status word of the current
 * device.  Every pipeline wait inside the kernels is bounded; a wait that runs
 * out records a nonzero code here (the first one wins) and the kernel winds down
 * without hanging.  While the word is nonzero, later launches on that device
 * return at once without computing.  This call synchronises the device, returns
 * FA2_OK if the word is zero and FA2_ERR_DEVICE_TIMEOUT otherwise (or
 * FA2_ERR_CUDA if it cannot be read), stores the raw word in *raw_code when
 * raw_code is not NULL, and clears the word when `reset` is nonzero.
 */
int fa2_device_status(int reset, int* raw_code);

/*
 * fa2_selftest_wait_timeout -- exercises the failure path.  Launches one thread
 * on `stream` that waits, with the same bounded wait every pipeline wait of the
 * kernels uses, on a barrier that nothing completes; after limit_ms (1..2000) it
 * gives up and records code 99 in the device status word, as a kernel whose
 * pipeline stalled would.  Nothing hangs and the context stays usable: later
 * launches see the word and return without computing until fa2_device_status
 * clears it.  A test hook; the pages have no counterpart.  Returns FA2_OK when
 * launched, FA2_ERR_SHAPE for limit_ms out of range.
 */
int fa2_selftest_wait_timeout(int limit_ms, void* stream);

/*
 * fa2_probe_ex2 -- throughput probe of the base-2 exponential of the special-
 * function pipe (the ex2 the softmax of both passes is built on; the pages'
 * "Writing FlashAttention 2 in Triton", Step 5, swaps exp for exp2 for this
 * reason).  Launches `blocks` CTAs of 256 threads on `stream`; every thread runs
 * 8 independent chains of `iters` steps, each step one ex2 and one add, and
 * writes one float to out[blocks * 256] (device, caller-owned, 4-byte aligned).
 * The caller times the launch: exponentials = blocks * 256 * 8 * iters.  A
 * measurement aid only; no result of the attention path depends on it.
 * Returns FA2_OK when launched, FA2_ERR_NULL, FA2_ERR_SHAPE (blocks outside
 * 1..65536 or iters outside 1..2^20), FA2_ERR_ALIGN, FA2_ERR_ARCH or
 * FA2_ERR_CUDA.
 */
int fa2_probe_ex2(float* out, int blocks, int iters, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA2_GB300_H */
