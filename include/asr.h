/*
 * asr.h -- C ABI of the GB300 fused AdamW step with Philox-keyed stochastic
 * rounding to bf16 (library: stochastic_rounding_gb300/libasr.so).
 *
 * What the operations compute is fixed by two pages:
 *   "Add stochastic rounding and philox RNG helpers" (FlyDSL PR 907),
 *       section Primitives -- stochastic rounding f32 -> bf16 and the Philox
 *       4x32 counter-based generator that feeds it;
 *   "adamw-sr", introduction and sections Method / Correctness -- one fused
 *       AdamW (Adam with decoupled weight decay) pass with bf16 parameters
 *       written back by stochastic rounding, its
 *       randomness keyed by (seed, step) and indexed by each element's global
 *       parameter position, identical whole or in shards with a base_index.
 *
 * Conventions shared by every entry point
 *   - Buffer pointers are DEVICE pointers (anything a kernel can dereference:
 *     cudaMalloc / torch CUDA memory, managed memory), owned by the caller.
 *     The kernels run on the calling thread's current device, so every
 *     buffer of a call must be memory that device can reach (its own, or a
 *     peer's with peer access enabled); the library cannot check this.
 *     The library allocates no device memory at run time (host scratch:
 *     asr_adamw_sr_multi_tensor may take a host buffer of two descriptors
 *     per tensor for the duration of the call; the static variant below
 *     takes none).  What it keeps between
 *     calls: per-device caches of launch shapes (and the tensor-map encoder's
 *     address), a 4-byte device error word with 64 four-byte copy slots
 *     (one per asr_take_device_error in progress) and the static
 *     descriptor array of
 *     asr_adamw_sr_multi_tensor_static.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising the host.  Buffers
 *     must stay valid until the stream reaches the work.
 *   - Arguments are checked before anything is launched.  A bad argument
 *     returns ASR_ERR_INVALID_VALUE / ASR_ERR_UNSUPPORTED_DTYPE and launches
 *     nothing.  A launch the CUDA runtime rejects returns ASR_ERR_CUDA (the
 *     CUDA error code is then available from asr_last_cuda_error()).  Faults
 *     that happen later on the GPU surface, as usual, at the next
 *     synchronising CUDA call of the caller.
 *   - n == 0 is a valid no-op (pointers may then be NULL).
 *   - The element-wise entry points (Philox, rounding, AdamW) accept any
 *     element alignment.  The AdamW step takes 128-bit vector paths for
 *     every tensor whose buffers are 16-byte aligned, and for the part of a
 *     tensor from its first element at which all four buffers are (the few
 *     elements before that take scalar units): the pipelined kernel, except
 *     that tensors launched together whose step moves at most 128 MiB (and
 *     whose base indices are multiples of 4 where random bits are drawn)
 *     take the register kernel, which starts faster.  A base_index that is
 *     not a multiple of 4 costs one more Philox call per 8 elements, as it
 *     does on the rounding op's vectorised path.  Every path gives the same
 *     bits.  The GEMM states its own requirements.
 *   - Buffers of one call must not overlap each other (not checked).
 *   - The library is thread-safe; calls on different streams may run
 *     concurrently on disjoint buffers.  One exception:
 *     asr_adamw_sr_multi_tensor_static keeps its table in one shared device
 *     array, so its calls must not overlap one another on the GPU.
 *   - CUDA graphs: asr_philox4x32, asr_stochastic_round_bf16,
 *     asr_adamw_sr_step, asr_adamw_sr_multi_tensor and asr_gemm_bf16_sr may
 *     be captured into a graph (stream capture) once a call of the same
 *     entry point with work to do has run on the device outside any capture
 *     -- that first call sets up the launch shapes of every kernel the entry
 *     point may pick on that device (for the two AdamW entry points, of
 *     both), so the captured calls need no set-up whatever their dtypes,
 *     alignment and sizes -- and a replay gives the bits the direct calls
 *     give.  asr_take_device_error waits for its
 *     stream and is not for capture; asr_take_device_error_async is.
 *   - The kernels are built for sm_103a (GB300) only; on any other GPU the
 *     first launch fails and the call returns ASR_ERR_CUDA.
 *
 * Random bits.  Philox4x32-10 (Salmon et al., SC'11; the generator cuRAND
 * calls Philox4_32_10): multipliers 0xD2511F53 and 0xCD9E8D57, Weyl
 * increments 0x9E3779B9 and 0xBB67AE85.  For an element with global index i at
 * (seed, step): key = (seed lo32, seed hi32), counter = ((i>>2) lo32,
 * (i>>2) hi32, step, 0); the element uses word (i & 3) of the four output
 * words, and only that word's low 16 bits.  One counter serves four
 * consecutive elements.
 *
 * bf16 values are passed as their 16-bit patterns (uint16_t), bf16 = the top
 * half of the binary32 pattern.
 */
#ifndef ASR_H
#define ASR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers (same underlying type). */
typedef struct CUstream_st *asr_stream_t;

typedef enum {
    ASR_OK = 0,
    ASR_ERR_INVALID_VALUE = 1,      /* NULL pointer with n > 0, step == 0,
                                       bad hyperparameter, bad count/size   */
    ASR_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype / rounding enum out of range    */
    ASR_ERR_CUDA = 3                /* the CUDA runtime rejected a call      */
} asr_status;

typedef enum { ASR_F32 = 0, ASR_BF16 = 1 } asr_dtype;

/* How a bf16 parameter is written back.  Ignored for f32 parameters. */
typedef enum {
    ASR_ROUND_SR = 0,   /* stochastic: add 16 Philox bits, truncate (default) */
    ASR_ROUND_RNE = 1   /* round to nearest, ties to even (biased baseline)   */
} asr_rounding;

/* AdamW hyperparameters of one step ("adamw-sr", Usage; Loshchilov and
 * Hutter 2019).  Requirements: lr, eps, weight_decay finite and >= 0;
 * 0 <= beta1, beta2 < 1; step >= 1 (the 1-based step count used both for the
 * bias corrections and as Philox counter word 2). */
typedef struct {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    uint32_t step;
    uint32_t rounding;      /* asr_rounding */
    uint64_t seed;
} asr_adamw_hparams;

/* The binary32 per-step scalars every element uses, each computed in binary64
 * from the hyperparameters and rounded once:
 *   b1 = beta1, b2 = beta2, eps, decay = 1 - lr*wd, omb1 = 1 - beta1,
 *   omb2 = 1 - beta2, step_size = lr / (1 - beta1^step),
 *   bc2s = sqrt(1 - beta2^step). */
typedef struct {
    float b1, b2, eps, decay, omb1, omb2, step_size, bc2s;
} asr_adamw_scalars;

/* One tensor (or one shard of a tensor) of a multi-tensor step. */
typedef struct {
    void *param;            /* n elements of param_dtype, updated in place   */
    const void *grad;       /* n elements of grad_dtype, read only           */
    float *exp_avg;         /* n binary32, first moment, updated in place    */
    float *exp_avg_sq;      /* n binary32, second moment, updated in place   */
    uint64_t n;
    uint64_t base_index;    /* global parameter position of element 0        */
    int32_t param_dtype;    /* asr_dtype */
    int32_t grad_dtype;     /* asr_dtype */
} asr_tensor_desc;

/* Philox4x32-10 words ("Add stochastic rounding and philox RNG helpers",
 * Primitives: philox_4x32(counter, key)).
 * For j in [0, n_ctr): counter = ((ctr_base + j) lo32, (ctr_base + j) hi32,
 * ctr2, ctr3), key = (seed lo32, seed hi32); out[4*j + w] = output word w.
 * out: device, 4*n_ctr uint32 (caller-owned). */
asr_status asr_philox4x32(uint32_t *out, uint64_t n_ctr, uint64_t ctr_base, uint32_t ctr2,
                          uint32_t ctr3, uint64_t seed, asr_stream_t stream);

/* Stochastic rounding f32 -> bf16 ("Add stochastic rounding and philox RNG
 * helpers", Primitives: stochastic_round_bf16(x, rand)).
 * out[j] = top 16 bits of (bits(x[j]) + (r_j & 0xFFFF)), where r_j is the
 * Philox word of global index base_index + j at (seed, step), or rbits[j]
 * when rbits is not NULL.  A NaN input gives (bits >> 16) | 0x0040 (still a
 * NaN, quiet); +-Inf are unchanged; finite values that round past the largest
 * bf16 become +-Inf.
 * x: device, n binary32.  rbits: device, n uint32, or NULL.  out: device, n
 * uint16 bf16 patterns. */
asr_status asr_stochastic_round_bf16(const float *x, const uint32_t *rbits, uint16_t *out,
                                     uint64_t n, uint64_t base_index, uint32_t step,
                                     uint64_t seed, asr_stream_t stream);

/* The per-step scalars of a hyperparameter set (host only; launches
 * nothing).  Returns ASR_ERR_INVALID_VALUE for a set the step would reject. */
asr_status asr_adamw_prepare(const asr_adamw_hparams *hp, asr_adamw_scalars *out);

/* One fused AdamW step on one tensor or shard ("adamw-sr", introduction and
 * Method).  For j in [0, n), with i = base_index + j and the scalars of
 * asr_adamw_prepare, in binary32 with every operation rounded on its own in
 * this order:
 *   p1  = p*decay;  m' = b1*m + omb1*g;  v' = b2*v + omb2*(g*g);
 *   den = sqrt(v')/bc2s + eps;  pn = p1 - step_size*(m'/den);
 * then m <- m', v <- v', and p <- pn (f32 param) or the bf16 rounding of pn
 * (stochastic with element i's Philox bits, or RNE, per hp->rounding).
 * param: device, n elements of pdt.  grad: device, n elements of gdt.
 * exp_avg / exp_avg_sq: device, n binary32 each.  hp: host. */
asr_status asr_adamw_sr_step(void *param, int32_t pdt, const void *grad, int32_t gdt,
                             float *exp_avg, float *exp_avg_sq, uint64_t n,
                             uint64_t base_index, const asr_adamw_hparams *hp,
                             asr_stream_t stream);

/* The same step over many tensors in one launch per dtype combination
 * (and kernel path) ("adamw-sr", Method: one global parameter position per
 * element).  Bitwise equal to calling asr_adamw_sr_step on each descriptor in
 * turn.  table: HOST array of n_tensors descriptors (read during the call
 * only); n_tensors >= 0.  Descriptors with n == 0 are skipped. */
asr_status asr_adamw_sr_multi_tensor(const asr_tensor_desc *table, int32_t n_tensors,
                                     const asr_adamw_hparams *hp, asr_stream_t stream);

/* The same step as asr_adamw_sr_multi_tensor, for callers that must not
 * allocate device memory: code running where another allocator owns the
 * device's memory (a framework's pooling allocator, a memory-capped job), so
 * that a raw cudaMalloc would fail or escape that allocator's accounting, and
 * code that must not pay for an allocation inside a training step.  The
 * pages have no counterpart: this is a packaging variant of the step.
 *
 * Its scratch, the descriptor table the kernel walks, is staged in a
 * library-owned static device array of ASR_STATIC_TABLE_MAX descriptors
 * (224 KB, held on every device that loads the library until the process
 * exits) instead of the launch parameters, so one launch per dtype group
 * covers up to ASR_STATIC_TABLE_MAX tensors.  Results are bitwise equal to
 * asr_adamw_sr_multi_tensor.
 *   - n_tensors > ASR_STATIC_TABLE_MAX returns ASR_ERR_INVALID_VALUE before
 *     anything is launched; otherwise the checks of the other entry points.
 *   - Allocates nothing: no cudaMalloc/cudaFree and no allocating library
 *     routine; host staging uses fixed static buffers.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with the device current); the first call that
 *     takes each of its kernels sets up that kernel's launch shape.
 *   - The table is copied into the array from the library's (pageable)
 *     host staging buffer with an asynchronous copy on `stream`: the runtime
 *     has taken the host bytes by the time the call returns, and the copy is
 *     ordered after earlier work on `stream` and before the kernels that
 *     read it.  The call does not wait for the GPU.
 *   - Every call reuses the one array and leaves its table there: calls whose
 *     kernels overlap on the GPU (other streams, other host threads) race on
 *     it.  Each call rewrites the part it uses; nothing has to start at zero. */
#define ASR_STATIC_TABLE_MAX 4096
asr_status asr_adamw_sr_multi_tensor_static(const asr_tensor_desc *table, int32_t n_tensors,
                                            const asr_adamw_hparams *hp, asr_stream_t stream);

/* bf16 GEMM with a stochastic-rounding epilogue on the tensor cores ("Add
 * stochastic rounding and philox RNG helpers", Consumer: the page's first
 * user of the rounding is a bf16 matrix product whose binary32 sums may be
 * written out by stochastic rounding, with random bits chosen per output
 * element from a seed, as an alternative to the default nearest rounding).
 * C = A . B^T with A: m x k, B: n x k, C: m x n, all row-major bf16 patterns
 * (device, caller-owned); f32 accumulation.  Output element (i, j) is
 * rounded from its f32 accumulator acc(i, j) exactly as
 * asr_stochastic_round_bf16 rounds element i*n + j with base_index 0 at
 * (seed, step) (rounding = ASR_ROUND_SR), or to nearest-even
 * (ASR_ROUND_RNE).  c_f32 (device, m x n f32, may be NULL) receives acc.
 * Requirements: n a multiple of 16, k a multiple of 8 (and k >= 8), m, n, k
 * at most 2^24, fewer than 2^31 output tiles (ceil(m/256) * ceil(n/256)),
 * all pointers 16-byte aligned; otherwise ASR_ERR_INVALID_VALUE before any
 * launch.  m == 0 or n == 0 is a no-op.
 * The summation order of acc is the tensor cores', so acc is reproducible
 * run to run on one GPU model but not bitwise equal to a CPU sum.  Runs on
 * clusters of two CTAs (tcgen05 cta_group::2) where the GPU can hold them,
 * else on one CTA per tile; the rounding of acc is the same either way. */
asr_status asr_gemm_bf16_sr(const uint16_t *a, const uint16_t *b, uint16_t *c, float *c_f32, uint64_t m,
                            uint64_t n, uint64_t k, uint32_t rounding, uint32_t step, uint64_t seed,
                            asr_stream_t stream);

/* Static description of a status code. */
const char *asr_status_string(asr_status status);

/* The CUDA runtime error code (cudaError_t as int) behind the calling
 * thread's most recent ASR_ERR_CUDA, 0 if none. */
int asr_last_cuda_error(void);

/* Sticky error bits raised on the device by the current device's kernels,
 * read and cleared in one atomic step.  Bit 0 (1): a pipeline wait inside a
 * kernel gave up after its time limit (2 s); the kernel then left the
 * affected tiles unfinished and returned instead of hanging.  Enqueues the
 * read on `stream`, waits for the stream, then stores the bits (0 = no
 * error) in *bits (host). */
asr_status asr_take_device_error(uint32_t *bits, asr_stream_t stream);

/* The same as asr_take_device_error without waiting (no counterpart on the
 * pages): enqueues on `stream` one thread that atomically reads and clears
 * the current device's error bits and writes them to *bits, and returns.
 * *bits holds the value once the stream has reached that point (wait for an
 * event recorded after the call).  bits: 4-byte aligned memory the GPU can
 * write -- device or managed memory of the current device, or page-locked
 * host memory (cudaHostAlloc / cudaMallocHost / cudaHostRegister); any other
 * pointer (pageable host memory, NULL) returns ASR_ERR_INVALID_VALUE and
 * launches nothing. */
asr_status asr_take_device_error_async(uint32_t *bits, asr_stream_t stream);

/* A tensor for asr_adamw_sr_multi_tensor_host: its device buffers (dev: the
 * step updates dev.param, dev.exp_avg and dev.exp_avg_sq in place and reads
 * the gradient from dev.grad) and its host side: grad_host, n elements of
 * dev.grad_dtype in page-locked host memory, copied into dev.grad before the
 * step; param_host, n elements of dev.param_dtype in page-locked host
 * memory that receives the updated parameters after the step, or NULL to
 * leave them on the device only. */
typedef struct {
    asr_tensor_desc dev;
    const void *grad_host;
    void *param_host;
} asr_host_tensor_desc;

/* The multi-tensor step for callers whose gradients arrive in host memory
 * and whose updated parameters go back to it (no counterpart on the pages:
 * a runtime around the step).  The tensors, in table order, are grouped into
 * chunks of consecutive tensors of at most chunk_elems elements (a larger
 * tensor is a chunk of its own; chunk_elems 0 means 2^28); for each chunk
 * the gradients are copied in on copy_in, the chunk's step runs on stream
 * once they have arrived (bitwise the step asr_adamw_sr_multi_tensor gives
 * the same descriptors), and its parameters are copied out on copy_out once
 * its step is done, so that with three distinct non-blocking streams the
 * copies of one chunk overlap the steps of its neighbours.  Ordering: all
 * of it follows the work queued on `stream` before the call, and the steps
 * also follow the work queued on copy_out before it (so a step never
 * overwrites parameters that an earlier call is still copying out); work
 * queued on `stream` after the call follows the steps -- and so the copies
 * in: the host gradients may then be overwritten -- while the copies out
 * complete on copy_out: wait on copy_out (an event recorded there after the
 * call, or a synchronisation) before reading the host parameters.  Not
 * joining copy_out back into `stream` lets one call's first copies in run
 * while the previous call's last copies out finish.  copy_in and copy_out
 * may be `stream` itself (no overlap then).  One copy
 * (cudaMemcpyAsync) per tensor and direction, except that consecutive
 * tensors of a chunk whose host and device ranges both follow on from one
 * another are copied together.  Host buffers must be page-locked
 * (cudaHostAlloc / cudaMallocHost / cudaHostRegister; checked with
 * cudaPointerGetAttributes -- any other pointer returns
 * ASR_ERR_INVALID_VALUE before anything is queued) and stay valid and
 * unchanged until the copies have run; the device gradient buffers must not
 * be in use by other work.  The library keeps a pool of CUDA events per
 * device for the ordering (created on first use, reused; at most 4,096 kept
 * per device, two per chunk are needed during a call).  Host scratch: a
 * descriptor array per call.  On ASR_ERR_CUDA part of the work may have been
 * queued. */
asr_status asr_adamw_sr_multi_tensor_host(const asr_host_tensor_desc *table, int32_t n_tensors,
                                          const asr_adamw_hparams *hp, uint64_t chunk_elems,
                                          asr_stream_t stream, asr_stream_t copy_in, asr_stream_t copy_out);

/* Kinds of kernel launch counted by asr_kernel_launches. */
typedef enum {
    ASR_KERNEL_ADAMW_SCALAR = 0,             /* AdamW, register kernel, scalar units */
    ASR_KERNEL_ADAMW_VECTOR = 1,             /* AdamW, register kernel, 128-bit units */
    ASR_KERNEL_ADAMW_PIPELINED = 2,          /* AdamW, pipelined kernel, two counters per unit */
    ASR_KERNEL_ADAMW_PIPELINED_ANY_BASE = 3, /* AdamW, pipelined kernel, three counters per unit */
    ASR_KERNEL_ADAMW_STATIC = 4,             /* AdamW through asr_adamw_sr_multi_tensor_static */
    ASR_KERNEL_ROUND = 5,                    /* asr_stochastic_round_bf16 */
    ASR_KERNEL_PHILOX = 6,                   /* asr_philox4x32 */
    ASR_KERNEL_GEMM = 7,                     /* asr_gemm_bf16_sr */
    ASR_KERNEL_KINDS = 8
} asr_kernel_kind;

/* Diagnostic (no counterpart on the pages): copies into counts[k], for
 * k < min(n, ASR_KERNEL_KINDS), how many kernels of kind k (asr_kernel_kind)
 * the library has launched in this process -- on every device, stream and
 * host thread, since it was loaded.  A launch is counted on the host when it
 * has been queued without error, so a launch captured into a CUDA graph
 * counts once and its replays do not.  Which AdamW kernel a step takes
 * depends on its buffers' alignment, base indices and size (see the
 * conventions above); these counters show which ones ran.  Makes no CUDA
 * call.  counts may be NULL only when n == 0; n < 0 returns
 * ASR_ERR_INVALID_VALUE. */
asr_status asr_kernel_launches(uint64_t *counts, int32_t n);

/* Diagnostic (no counterpart on the pages): launches one thread that waits,
 * with the kernels' bounded-wait routine and a limit of limit_ns
 * (1 .. 2e9 ns), on a barrier nothing arrives on.  The wait gives up, the
 * kernel returns, and the next asr_take_device_error reports bit 0.  Used to
 * show that a stuck pipeline ends with a status instead of a hang. */
asr_status asr_selftest_wait_timeout(uint64_t limit_ns, asr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ASR_H */
