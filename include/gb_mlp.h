/*
 * gb_mlp.h - C ABI of the tensor-sliced transformer MLP block (forward, backward,
 * fp32 gradient accumulation) on one GB300 GPU (sm_103a).
 *
 * The operation (Megatron tensor-parallel MLP, "STRONGHOLD: Fast and Affordable
 * Billion-scale Deep Learning Model Training", slides items 7-8; gradient
 * accumulation over micro-batches, "Using DeepSpeed and Megatron to Train
 * Megatron-Turing NLG 530B", Key points):
 *
 *   A [h, ffn] is split column-wise into t slices A_i = A[:, i*f:(i+1)*f], f = ffn/t
 *   B [ffn, h] is split row-wise    into t slices B_i = B[i*f:(i+1)*f, :]
 *   forward   U_i = X A_i + a_i,  Y_i = GeLU(U_i),  Z = sum_i Y_i B_i   (operator g)
 *             O   = R + dropout(Z + b)
 *   backward  dZ = dO * m / (1-p),  db += sum_tok dZ
 *             dU_i = (dZ B_i^T) * GeLU'(U_i),  da_i += sum_tok dU_i
 *             dB_i += Y_i^T dZ,  dA_i += X^T dU_i
 *             dX = [dO +] sum_i dU_i A_i^T                               (operator f)
 *
 * Every slice runs on this GPU; the sums over slices that the pages perform with
 * all-reduces across GPUs are on-device fp32 reductions here.
 *
 * GeLU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).  Dropout
 * is inverted dropout: element e = (token_offset + token) * h + column of the
 * [tokens, h] output is kept iff (SplitMix64(seed, e) >> 32) >= round(p * 2^32),
 * where SplitMix64(seed, e) is output number e of a SplitMix64 stream seeded with
 * `seed` (Steele, Lea & Flood, OOPSLA 2014), and kept values are scaled by
 * 1/(1-p).  The mask does not depend on t, the slice, or any value.
 *
 * Conventions for every entry point:
 *   - Tensors are row-major and contiguous; mlp_bf16 is the raw bit pattern of a
 *     bfloat16.  Shapes: X, R, O, dO, dX, dZ [tokens, h]; U, Y, dU [tokens, ffn];
 *     A [h, ffn]; a [ffn]; B [ffn, h]; b [h]; dA [h, ffn]; da [ffn]; dB [ffn, h];
 *     db [h]; Zacc, dXacc [tokens, h] fp32.
 *   - All pointers are DEVICE pointers owned by the caller, 16-byte aligned.  No
 *     call allocates device memory.  The library's own device memory is static
 *     module memory, held by every GPU that loads the library until the process
 *     exits: the 2-word status word; the split-tail partial sums and arrival
 *     counters of the GEMMs (4 regions of 304 x 2 x 32 x 256 fp32, about 20 MB
 *     each, see mlp_set_split_tail); the tile counters of the GEMMs' dynamic
 *     scheduler (2 ints per region, see mlp_set_tile_scheduler); and the 16 MiB
 *     fp32 array of mlp_fwd_static_scratch.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and runs asynchronously.  A nonzero return means nothing was enqueued,
 *     except MLP_ECUDA, which reports a failed launch (later launches of the same
 *     call are not attempted).  mlp_last_error() describes the failure.
 *   - Constraints: h > 0, h % 8 == 0; ffn % t == 0, f = ffn/t, f % 8 == 0;
 *     0 < tokens < 2^31; 0 <= p < 1; -1 <= slice < t.
 *   - A kernel that detects a broken pipeline (a bounded wait that ran out)
 *     records MLP_ETIMEOUT in the device status word and returns;
 *     mlp_sync_status() reports it.
 */
#ifndef GB_MLP_H
#define GB_MLP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mlp_bf16; /* raw bfloat16 bits */

enum {
  MLP_OK = 0,
  MLP_EINVAL = -1,       /* a size, count or probability out of range, or a NULL pointer */
  MLP_EALIGN = -2,       /* a pointer not 16-byte aligned */
  MLP_EUNSUPPORTED = -3, /* no sm_103a device, or a shape the kernels do not take */
  MLP_ECUDA = -4,        /* a CUDA call or launch failed */
  MLP_ETIMEOUT = -5      /* a kernel gave up on a bounded wait (device status word) */
};

/*
 * mlp_fwd - forward of one micro-batch (STRONGHOLD slides, items 7-8).
 *
 *   slice == -1: all t slices inside this call.  Each GEMM launch covers every
 *                slice: the first walks the column blocks A_0 .. A_{t-1}, the
 *                second's reduction loop walks the row blocks B_0 .. B_{t-1}, so
 *                the sum over slices is formed in the fp32 accumulator on chip.
 *                Zacc is not used (may be NULL).
 *   slice == i : slice i only.  Calls must come in order i = 0 .. t-1 on one
 *                stream; slice 0 overwrites Zacc, slices 0 .. t-2 accumulate
 *                into it (fp32, in HBM), and slice t-1 writes O.
 *   X      [tokens, h]   input activations.
 *   A, a   [h, ffn], [ffn]   first weight and bias (slice i = columns i*f ..).
 *   B, b   [ffn, h], [h]     second weight and bias (slice i = rows i*f ..).
 *   R      [tokens, h]   residual; NULL means R = X.
 *   U, Y   [tokens, ffn] outputs: pre-activation and GeLU output (bf16), kept
 *                        for the backward; slice i writes columns i*f .. .
 *   Zacc   [tokens, h] fp32 workspace for the sum over slices of one-slice
 *                        calls; may be NULL when t == 1 or slice == -1.
 *   O      [tokens, h]   output, written by the last slice.
 * Returns MLP_OK or an error code.
 */
int mlp_fwd(int h, int ffn, int t, int slice, int64_t tokens, float p, uint64_t seed, uint64_t token_offset,
            const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a, const mlp_bf16* B, const mlp_bf16* b,
            const mlp_bf16* R, mlp_bf16* U, mlp_bf16* Y, float* Zacc, mlp_bf16* O, void* stream);

/*
 * mlp_bwd - backward of one micro-batch.  Weight and bias gradients go to the
 * fp32 dA, da, dB, db: with accumulate = 1 they are ADDED (+=), which sums the
 * micro-batches of a step (gradient accumulation); with accumulate = 0 they
 * OVERWRITE the accumulators, which is how the first micro-batch of a step starts
 * the sum without a separate grad_accum_reset (the two agree bit for bit:
 * 0 + x = x).
 *
 *   slice == -1 or slice == i as for mlp_fwd (order 0 .. t-1).  The call with
 *   slice 0 (or -1) computes dZ and db; the call with slice t-1 (or -1) writes
 *   dX.  With slice == -1 the sum over slices of dU_i A_i^T is formed in the
 *   fp32 accumulator on chip and dXacc is not used.
 *   residual_grad  1: dX = dO + sum_i dU_i A_i^T (the residual R was X);
 *                  0: dX = sum_i dU_i A_i^T.
 *   accumulate     1: dA, da, dB, db += this micro-batch's gradients;
 *                  0: dA, da, dB, db  = this micro-batch's gradients.  With
 *                     one-slice calls each slice writes its own columns of dA
 *                     and da and rows of dB; db is written by the slice-0 call.
 *   dO     [tokens, h]  upstream gradient of O.
 *   X, A, B           as passed to mlp_fwd; U, Y as written by mlp_fwd.
 *   dZ     [tokens, h]  workspace/output: gradient after dropout (bf16).
 *   dU     [tokens, ffn] workspace/output: gradient of the pre-activation (bf16).
 *   dXacc  [tokens, h] fp32 workspace for the sum over slices of one-slice
 *                        calls; may be NULL when t == 1 or slice == -1.  In
 *                        those calls a non-NULL dXacc serves instead as scratch
 *                        for transposed bf16 copies of X and dZ that speed up
 *                        the weight-gradient GEMMs (mlp_set_wgrad_transpose);
 *                        either way its contents are undefined afterwards.
 *   dX     [tokens, h]  output (overwritten).
 *   dA, da, dB, db    fp32 gradient accumulators (+= or =, see accumulate).
 * Returns MLP_OK or an error code.
 */
int mlp_bwd(int h, int ffn, int t, int slice, int64_t tokens, float p, uint64_t seed, uint64_t token_offset,
            int residual_grad, int accumulate, const mlp_bf16* dO, const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B,
            const mlp_bf16* U, const mlp_bf16* Y, mlp_bf16* dZ, mlp_bf16* dU, float* dXacc, mlp_bf16* dX,
            float* dA, float* da, float* dB, float* db, void* stream);

/*
 * grad_accum_reset - zero the fp32 gradient accumulators dA [h, ffn], da [ffn],
 * dB [ffn, h], db [h] before the first micro-batch of a step (gradient
 * accumulation, MT-NLG summary page, Key points).  Returns MLP_OK or an error.
 */
int grad_accum_reset(int h, int ffn, float* dA, float* da, float* dB, float* db, void* stream);

/*
 * adam_step - one mixed-precision Adam update (decoupled weight decay) of n
 * parameters from their fp32 gradient accumulator.  The pages give the cost of
 * mixed-precision Adam, about 20 bytes of training state per parameter ("Using
 * DeepSpeed and Megatron to Train Megatron-Turing NLG 530B", Key points); the
 * update is the published algorithm (Kingma & Ba 2015; Loshchilov & Hutter 2019):
 *   g = grad * grad_scale;  m = beta1 m + (1-beta1) g;  v = beta2 v + (1-beta2) g^2
 *   master = master (1 - lr weight_decay) - lr/(1-beta1^step) m / (sqrt(v/(1-beta2^step)) + eps)
 *   weight = bf16(master)   (round to nearest even)
 * grad [n] fp32 (read only), master, m, v [n] fp32 (updated in place), weight [n]
 * bf16 (written): device pointers; grad, master, m, v 16-byte aligned, weight
 * 8-byte aligned.  step >= 1 counts updates; 0 <= beta1, beta2 < 1; eps > 0;
 * lr, weight_decay >= 0.  Returns MLP_OK or an error code (nothing enqueued).
 */
int adam_step(int64_t n, const float* grad, float grad_scale, float* master, float* m, float* v, mlp_bf16* weight,
              float lr, float beta1, float beta2, float eps, float weight_decay, int step, void* stream);

/*
 * attn_fwd - forward of the tensor-sliced self-attention block (the next row after
 * the MLP block).  The pages give the model as a left-to-right decoder with 128
 * heads trained with Megatron tensor slicing (jiqizhixin article on MT-NLG; MT-NLG
 * summary page); they spell the split out only for the MLP ("STRONGHOLD" slides,
 * items 7-8).  Reading, mirroring it: the fused QKV projection is split
 * column-wise by heads, each head attends causally within its sequence, and the
 * output projection is split row-wise with the partial products summed over
 * slices (operator g), then bias, dropout and residual as in the MLP block:
 *   QKV = X Wqkv + bqkv;  per sequence and head: P = softmax(mask(Q K^T / sqrt(d))),
 *   O_head = P V;  out = R + dropout(O Wo + bo)        (the MLP block's dropout mask)
 * All t slices run in every call; each launch covers every head, and the sum over
 * slices of O_i Wo_i forms in the fp32 accumulator.
 *   h = hidden, nh = heads (d = h / nh, d % 8 == 0), t | nh, tokens = n_seq * seq_len,
 *   seq_len % 8 == 0.
 *   X, R, O, out [tokens, h]; Wqkv [h, 3h] = [Wq | Wk | Wv] with head j at columns
 *   j*d .. (j+1)*d of each block; bqkv [3h]; Wo [h, h]; bo [h]  (bf16).
 *   QKV [tokens, 3h] bf16 (saved), P [n_seq, nh, seq_len, seq_len] bf16 (saved
 *   probabilities, exact zeros above the diagonal), O [tokens, h] bf16 (saved),
 *   S: fp32 workspace of P's shape (not touched by the fused core, see
 *   mlp_set_attn_fused, but always required).
 * Returns MLP_OK or an error code.
 */
int attn_fwd(int h, int nh, int t, int64_t tokens, int seq_len, float p, uint64_t seed, uint64_t token_offset,
             const mlp_bf16* X, const mlp_bf16* Wqkv, const mlp_bf16* bqkv, const mlp_bf16* Wo, const mlp_bf16* bo,
             const mlp_bf16* R, mlp_bf16* QKV, float* S, mlp_bf16* P, mlp_bf16* O, mlp_bf16* out, void* stream);

/*
 * attn_bwd - backward of the attention block; dWqkv, dbqkv, dWo, dbo (fp32) are
 * added to (accumulate = 1) or overwritten (accumulate = 0), as in mlp_bwd:
 *   dZ = dOut m / (1-p); dbo = sum dZ; dWo = O^T dZ; dO = dZ Wo^T;
 *   per sequence and head: dV = P^T dO; dP = dO V^T; dS = P (dP - rowsum(dP P)) / sqrt(d);
 *   dQ = dS K; dK = dS^T Q;  dWqkv = X^T dQKV; dbqkv = sum dQKV;
 *   dX = [dOut +] dQKV Wqkv^T   (operator f; residual_grad selects the dOut term)
 * rowsum(dP P) is taken as rowsum(dO * O), the same quantity (P V = O), and dP is
 * never stored: the product dO V^T goes straight into dS in the GEMM's epilogue.
 * dZ, dO [tokens, h] and dS (P's shape) are bf16 workspaces (dS is written only in
 * the tiles on or below the causal diagonal that are read back, and may also hold
 * transposed copies of dZ and X, see mlp_set_wgrad_transpose),
 * dP an fp32 workspace of at least n_seq * nh * seq_len floats (the row sums),
 * dQKV [tokens, 3h] bf16, dX [tokens, h] bf16.  Returns MLP_OK or an error.
 */
int attn_bwd(int h, int nh, int t, int64_t tokens, int seq_len, float p, uint64_t seed, uint64_t token_offset,
             int residual_grad, int accumulate, const mlp_bf16* dOut, const mlp_bf16* X, const mlp_bf16* Wqkv,
             const mlp_bf16* Wo, const mlp_bf16* QKV, const mlp_bf16* P, const mlp_bf16* O, mlp_bf16* dZ,
             mlp_bf16* dO, float* dP, mlp_bf16* dS, mlp_bf16* dQKV, mlp_bf16* dX, float* dWqkv, float* dbqkv,
             float* dWo, float* dbo, void* stream);

/*
 * mlp_sync_status - synchronise `stream`, then return and clear the device status
 * word: MLP_OK, or MLP_ETIMEOUT if a kernel gave up on a bounded wait since the
 * last call (mlp_last_error() then names the wait), or MLP_ECUDA.
 */
int mlp_sync_status(void* stream);

/* mlp_last_error - thread-local description of the last nonzero return. */
const char* mlp_last_error(void);

/*
 * mlp_dropout_mask - the keep mask the forward and backward use, one byte per
 * element of the [tokens, h] output (1 = kept), written to device memory m.
 * For tests and inspection; the block itself never materialises the mask.
 */
int mlp_dropout_mask(int h, int64_t tokens, float p, uint64_t seed, uint64_t token_offset, uint8_t* m,
                     void* stream);

/*
 * mlp_gelu_probe - y[i] = GeLU(x[i]), dy[i] = GeLU'(x[i]) for n fp32 device
 * values, with the same device functions the GEMM epilogues use.  For tests.
 */
int mlp_gelu_probe(const float* x, int64_t n, float* y, float* dy, void* stream);

/*
 * mlp_wait_timeout_probe - launch one kernel that waits on a barrier nothing
 * arrives on, giving up after limit_ns nanoseconds, so that the next
 * mlp_sync_status() returns MLP_ETIMEOUT.  Tests the error path of bounded waits
 * without faulting or hanging the GPU.  limit_ns must be <= 10^9.
 */
int mlp_wait_timeout_probe(uint64_t limit_ns, void* stream);

/*
 * mlp_set_cta_pair - choose the GEMM variant for later calls in this process:
 * -1 (default) CTA pairs (clusters of two CTAs, 256 x 256 tiles, tcgen05
 * cta_group::2) whenever a GEMM has more than 128 rows, else single CTAs
 * (128 x 256 tiles); 0 always single CTAs; 1 always CTA pairs.  Results agree
 * within the fp32 summation-order tolerance.  Returns MLP_OK or MLP_EINVAL.
 */
int mlp_set_cta_pair(int mode);

/*
 * mlp_set_dependent_launch - enable (1, the default) or disable (0), for later
 * calls in this process, programmatic dependent launch: each kernel may be
 * scheduled while the previous kernel on its stream finishes, so its prologue
 * overlaps that kernel's tail; every kernel waits for the previous kernel's
 * results before it touches global memory, so results do not change.
 * Returns MLP_OK or MLP_EINVAL.
 */
int mlp_set_dependent_launch(int enable);

/*
 * mlp_set_split_tail - enable (1, the default) or disable (0), for later calls in
 * this process, the split tail of the GEMMs with a bf16 epilogue: when a GEMM's last
 * wave of output tiles would occupy at most half of the CTA pairs (CTAs), each of
 * those tiles is computed as two halves of its reduction by two pairs, whose fp32
 * partial sums are added (in either order: the sum is the same) before the
 * epilogue.  Results stay deterministic; they differ from the unsplit ones only by
 * fp32 summation order.  The partial sums use statically allocated device memory,
 * one 20 MB region per stream for the first 4 streams that launch such a GEMM;
 * GEMMs on further streams run unsplit.  Returns MLP_OK or MLP_EINVAL.
 */
int mlp_set_split_tail(int enable);

/*
 * mlp_set_wgrad_transpose - how mlp_bwd feeds the weight-gradient GEMMs
 * dB (+)= Y^T dZ and dA (+)= X^T dU, whose reduction runs over the tokens, so
 * that both operands of each are MN-major as stored (a GEMM with two MN-major
 * operands runs about 5 % slower than with one K-major operand), for later calls
 * in this process:
 *   1  whenever dXacc is free (t == 1 or slice == -1), passed and 16-byte
 *      aligned, tokens % 8 == 0 and tokens > 960, and both GEMMs run on CTA pairs
 *      (see mlp_set_cta_pair): one extra launch writes X^T and dZ^T
 *      ([h, tokens] bf16 each) into dXacc, and the two GEMMs read those copies as
 *      K-major operands;
 *  -1  (the default) the same, for GEMMs of at least 1e12 FLOP each (smaller ones
 *      do not repay the copies);
 *   0  never.
 * attn_bwd does the same for dWo (+)= O^T dZ and dWqkv (+)= X^T dQKV when seq_len
 * >= the head size: the copies dZ^T and X^T go to its dS workspace, which is free
 * before the attention core writes it and after the products read it.
 * The products and their reduction order are the same either way.  Returns
 * MLP_OK or MLP_EINVAL.
 */
int mlp_set_wgrad_transpose(int mode);

/*
 * mlp_set_attn_fused - choose, for later attn_fwd / attn_bwd calls in this
 * process, how the attention core runs: 1 (the default) fused kernels when the
 * head size d is at most 192, 0 the unfused launches.
 *   forward, fused: S = Q K^T / sqrt(d) stays in tensor memory; two passes over
 *     the key tiles, the first for each row's maximum and sum, the second writing
 *     the normalised bf16 P and accumulating O = P V; the S workspace is not used.
 *   forward, unfused: a batched GEMM writing S, the row softmax, a batched GEMM.
 *   backward, fused: per key tile, dP = dO V^T, dV += P^T dO, dS and dK += dS^T Q
 *     in one kernel, then dQ = dS K as a batched GEMM.
 *   backward, unfused: batched GEMMs for dV, dO V^T (with the dS epilogue), dQ, dK.
 * The two agree within a bf16 rounding step of P (the softmax sums run in another
 * order).  Returns MLP_OK or MLP_EINVAL.
 */
int mlp_set_attn_fused(int enable);

/*
 * mlp_set_tile_scheduler - the order in which the persistent GEMM kernels hand
 * out their output tiles, for later calls in this process: 0 static round-robin;
 * 1 dynamic, each CTA pair taking the next tile from a counter in global memory
 * when it is ready for one (this balances GEMMs whose tiles carry unequal work);
 * -1 (the default) dynamic for the batched causal attention products, static for
 * every other GEMM.  Results
 * are bit-identical either way (a tile's arithmetic does not depend on which CTA
 * computes it).  The counters are static device memory, one pair per stream
 * region (the regions of mlp_set_split_tail); GEMMs on a fifth stream, GEMMs of
 * one wave, and launches that overlap the previous kernel on their stream use the
 * static order.  Returns MLP_OK or MLP_EINVAL.
 */
int mlp_set_tile_scheduler(int mode);

/* mlp_launch_count - number of kernels this library has launched in this process. */
uint64_t mlp_launch_count(void);

/*
 * mlp_trace_begin - from now on, bracket every kernel this library launches with
 * a pair of CUDA events on the launch stream, for at most `capacity` launches
 * (later launches are not traced).  The events are created here (host-side
 * resources only).  Returns MLP_OK, or MLP_EINVAL if a trace is already running.
 */
int mlp_trace_begin(int capacity);

/*
 * mlp_trace_end - stop tracing, wait for the traced launches and report up to
 * max_entries of them in launch order: kinds[i] (0..5 = the GEMMs F1, F2, B2, B3,
 * B4, B5 of the forward/backward; 10 = dropout backward + db; 11 = column sum
 * for da; 12 = accumulator reset; 14 = adam_step; 15 = the transposed copies of
 * X and dZ (mlp_set_wgrad_transpose); 20 = attention GEMMs; 21 =
 * softmax forward / backward; 22 = fused attention core), mnk[3i..3i+2] = the
 * launch's M, N, K (GEMMs; for the fused core: query rows, keys per sequence, d)
 * or rows, columns, 0, and ms[i] = its device time in milliseconds.  Any output
 * pointer may be NULL.  Returns the number of entries written, or an error code.
 */
int mlp_trace_end(int max_entries, int* kinds, int64_t* mnk, float* ms);

/*
 * mlp_fwd_static_scratch - mlp_fwd for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is an integration variant.
 *
 * One-slice forward calls (slice = i with t > 1) sum the row-split partial
 * products of successive calls in an fp32 [tokens, h] workspace, which mlp_fwd
 * takes from the caller (Zacc).  A plugin that runs inside a host application
 * owning all device memory through its own pool, or a serving loop that must not
 * allocate once it runs (cudaMalloc / cudaFree can synchronise the device), has no
 * such buffer to give.  This entry point takes the same arguments as mlp_fwd
 * without Zacc and uses a fixed 16 MiB array in the library's own device memory
 * instead; every GPU that loads the library holds that array until the process
 * exits.  It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *
 *   - tokens * h must not exceed 4,194,304 (16 MiB of fp32), else MLP_EINVAL
 *     with a message naming the limit; the limit applies to every call.
 *   - The first call on a device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents.  The
 *     slice-0 call overwrites it (nothing needs clearing), later slices add to it,
 *     and the last slice reads it.  Calls whose work overlaps on the GPU (other
 *     streams, other threads, other sequences of one-slice calls) race on it.
 * Everything else (arguments, layouts, results) is as for mlp_fwd.
 */
int mlp_fwd_static_scratch(int h, int ffn, int t, int slice, int64_t tokens, float p, uint64_t seed,
                           uint64_t token_offset, const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a,
                           const mlp_bf16* B, const mlp_bf16* b, const mlp_bf16* R, mlp_bf16* U, mlp_bf16* Y,
                           mlp_bf16* O, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB_MLP_H */
