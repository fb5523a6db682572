/*
 * conv.h -- C ABI of the implicit-GEMM conv2d library for GB300 (sm_103a).
 *
 * One layer type: a 2-D convolution with no padding, a square K x K kernel,
 * stride S, NCHW activations, computed as an implicit GEMM on the GPU.  The
 * operations are the three of PufferLib PR #522 ("Speedups to
 * gemm_conv_forward and gemm_conv_backward kernels"; its bench blocks time a
 * "forward" with relu=1 on layer 1, and a "backward" made of "wgrad" and
 * "d_input"):
 *
 *   OH = floor((H - K) / S) + 1,   OW = floor((W - K) / S) + 1
 *   conv_fwd         y[b,oc,oh,ow]   = act(sum_{ic,kh,kw} x[b,ic,oh*S+kh,ow*S+kw] * w[oc,ic,kh,kw])
 *                    act = max(., 0) (result +0 for a non-positive sum) when relu, else identity
 *   g                = dy * [y > 0] when relu (y: the forward output), else dy
 *   conv_bwd_data    dx[b,ic,h,w]    = sum over (oc,kh,kw,oh,ow) with oh*S+kh = h, ow*S+kw = w
 *                                      of g[b,oc,oh,ow] * w[oc,ic,kh,kw]
 *   conv_bwd_filter  dw[oc,ic,kh,kw] = sum_{b,oh,ow} g[b,oc,oh,ow] * x[b,ic,oh*S+kh,ow*S+kw]
 *
 * and the layer's per-output-channel bias (the same PR's "n3_conv_bias_grad"
 * bench blocks time its gradient for both conv layers, conv1 with 12 output
 * positions and conv2 with 2, OC = 128, B = 32768):
 *
 *   conv_fwd_bias    y[b,oc,oh,ow]   = act(bias[oc] + sum_{ic,kh,kw} ... as conv_fwd)
 *   conv_bwd_bias    db[oc]          = sum_{b,oh,ow} g[b,oc,oh,ow]
 *
 * Layouts (dense, row-major, no strides): x, dx (B,IC,H,W); y, dy
 * (B,OC,OH,OW); w, dw (OC,IC,K,K); bias, db (OC).  Every tensor of a call has the
 * descriptor's dtype: CONV_F32 (binary32 in and out, fp32 arithmetic) or
 * CONV_BF16 (bfloat16 in and out, fp32 accumulation, one round-to-nearest-even
 * rounding of each result).
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers (cudaMalloc'd or equivalent) on the
 *     current CUDA device, owned by the caller; the library keeps no reference
 *     after the call returns.  Base pointers must be 16-byte aligned.  Outputs
 *     must not overlap inputs.
 *   - Memory: no entry point allocates.  conv_fwd, conv_fwd_bias, conv_bwd_data
 *     and conv_bwd_bias use no memory beyond their arguments (their kernels
 *     format the weights on chip and reduce split sums inside thread-block
 *     clusters through distributed shared memory); conv_fwd_ws,
 *     conv_bwd_data_ws and conv_bwd_filter use a workspace the caller sizes with
 *     the matching *_workspace_size query and owns; conv_bwd_filter_noalloc uses
 *     a fixed array inside the library.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream): they
 *     enqueue kernels and return; they never synchronise.  Each call
 *     overwrites its whole output (it does not accumulate into it).
 *   - Results are deterministic: the same inputs give bit-identical outputs,
 *     run to run (fixed reduction orders, no floating-point atomics).
 *   - Errors are returned as a conv_status_t.  Argument errors are detected on
 *     the host before anything is enqueued; CONV_ERR_CUDA reports a failed
 *     launch (cudaGetLastError) and leaves the output unspecified.
 *   - A batch of B = 0 is valid: conv_fwd and conv_bwd_data do nothing;
 *     conv_bwd_filter writes dw = 0.
 *   - Index arithmetic is 32-bit: every tensor must hold fewer than 2^31
 *     elements (CONV_ERR_UNSUPPORTED otherwise).
 */
#ifndef IGCONV_CONV_H
#define IGCONV_CONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA include. */
struct CUstream_st;
typedef struct CUstream_st* conv_stream_t;

typedef enum { CONV_F32 = 0, CONV_BF16 = 1 } conv_dtype_t;

/* Shape descriptor.  relu is 0 or 1; dtype is a conv_dtype_t value. */
typedef struct {
    int32_t B, IC, OC, H, W, K, S, relu;
    int32_t dtype;
} conv_desc_t;

typedef enum {
    CONV_OK = 0,
    CONV_ERR_NULL = -1,        /* a required pointer is NULL                         */
    CONV_ERR_DESC = -2,        /* descriptor invalid: a dim < 1 (B < 0), H or W < K,
                                  relu not 0/1, dtype unknown                         */
    CONV_ERR_UNSUPPORTED = -3, /* valid but outside the library's limits (2^31)      */
    CONV_ERR_ALIGN = -4,       /* a base pointer is not 16-byte aligned              */
    CONV_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than the queried size    */
    CONV_ERR_CUDA = -6         /* a CUDA call or kernel launch failed                */
} conv_status_t;

/* Algorithm families (conv_set_algo / conv_query). */
typedef enum {
    CONV_ALGO_AUTO = 0,   /* library choice (default)                                 */
    CONV_ALGO_DIRECT = 1, /* one thread (bias grad: one warp) per output element; any
                             shape                                                    */
    CONV_ALGO_FFMA = 2,   /* fp32 CUDA-core tiled kernels: FFMA register-tiled
                             implicit GEMM; for the bias grad, the column-sum kernel  */
    CONV_ALGO_TC = 3      /* tcgen05 tensor cores, TMEM accumulator (bf16 operands,
                             or fp32 as three tf32 products)                          */
} conv_algo_t;

typedef enum {
    CONV_OP_FWD = 0, CONV_OP_BWD_DATA = 1, CONV_OP_BWD_FILTER = 2, CONV_OP_BWD_BIAS = 3,
    CONV_OP_FWD_WS = 4,      /* conv_fwd_ws / conv_fwd_bias with a workspace (conv_query only) */
    CONV_OP_BWD_DATA_WS = 5, /* conv_bwd_data_ws (conv_query only)                           */
    CONV_OP_BWD = 6          /* conv_bwd, the fused backward (conv_query only)              */
} conv_op_t;

/* Forward:  y = act(conv(x, w)).
 *   x: (B,IC,H,W)   w: (OC,IC,K,K)   y: (B,OC,OH,OW), written.
 * Returns CONV_OK or an error code (see above). */
int conv_fwd(const conv_desc_t* desc, const void* x, const void* w, void* y,
             conv_stream_t stream);

/* Forward with the per-channel bias:  y = act(conv(x, w) + bias), the bias
 * added in fp32 to the finished sum, before the activation and the one
 * rounding to the output dtype.  Same kernels, plans and conventions as
 * conv_fwd (conv_query / conv_set_algo with CONV_OP_FWD cover both).
 *   bias: (OC) in the descriptor's dtype, required (use conv_fwd for none). */
int conv_fwd_bias(const conv_desc_t* desc, const void* x, const void* w, const void* bias, void* y,
                  conv_stream_t stream);

/* The forward with a workspace: the same result as conv_fwd / conv_fwd_bias, bit for bit
 * (bias may be NULL: no bias).  With a workspace the tensor-core path first packs w once
 * into the operand tiles' exact shared-memory image (a small kernel), and the implicit GEMM
 * then fetches each tile with one bulk copy instead of formatting w in every CTA, which is
 * faster whenever the CTAs together would format w many times over (PufferLib PR #522's
 * layer-1 shape at B = 1024 and above).
 *   workspace: device buffer of at least conv_fwd_workspace_size(desc) bytes, 16-byte
 *   aligned, owned by the caller; contents on entry are ignored and on return are
 *   unspecified.  May be NULL when the size is 0 (then the call is conv_fwd's).
 *   CONV_ERR_WORKSPACE if it is NULL or smaller than the queried size. */
size_t conv_fwd_workspace_size(const conv_desc_t* desc);
int conv_fwd_ws(const conv_desc_t* desc, const void* x, const void* w, const void* bias, void* y,
                void* workspace, size_t workspace_bytes, conv_stream_t stream);

/* Data gradient (d_input):  dx = conv^T(g, w), g = dy masked by y > 0 when relu.
 *   dy: (B,OC,OH,OW)  w: (OC,IC,K,K)  y: (B,OC,OH,OW) forward output, required
 *   when desc->relu (the mask source), ignored otherwise (may be NULL)
 *   dx: (B,IC,H,W), written. */
int conv_bwd_data(const conv_desc_t* desc, const void* dy, const void* w, const void* y,
                  void* dx, conv_stream_t stream);

/* d_input with a workspace: the same result as conv_bwd_data, bit for bit; the tensor-core
 * path packs w^T once into the workspace (see conv_fwd_ws).
 *   workspace: at least conv_bwd_data_workspace_size(desc) bytes, 16-byte aligned, owned by
 *   the caller, contents ignored on entry and unspecified on return; may be NULL when the
 *   size is 0.  CONV_ERR_WORKSPACE if it is NULL or too small. */
size_t conv_bwd_data_workspace_size(const conv_desc_t* desc);
int conv_bwd_data_ws(const conv_desc_t* desc, const void* dy, const void* w, const void* y, void* dx,
                     void* workspace, size_t workspace_bytes, conv_stream_t stream);

/* Bytes of device workspace conv_bwd_filter needs for this descriptor on the
 * current device (split-K partial sums), or 0 if it needs none or the
 * descriptor is invalid.  Host-only; depends on the device's SM count. */
size_t conv_bwd_filter_workspace_size(const conv_desc_t* desc);

/* Weight gradient (wgrad):  dw = sum over b,oh,ow of g (x) patches(x), as a
 * split-K reduction over B*OH*OW: a first kernel writes fp32 partial sums of
 * contiguous ranges of (b,oh,ow) into the workspace, a second sums them in
 * ascending range order and rounds once to the output dtype.
 *   x: (B,IC,H,W)  dy: (B,OC,OH,OW)  y: forward output, required when relu
 *   dw: (OC,IC,K,K), written.
 *   workspace: device buffer of at least conv_bwd_filter_workspace_size(desc)
 *   bytes, 16-byte aligned, owned by the caller; contents on entry are
 *   ignored and on return are unspecified.  May be NULL when the size is 0. */
int conv_bwd_filter(const conv_desc_t* desc, const void* x, const void* dy, const void* y,
                    void* dw, void* workspace, size_t workspace_bytes, conv_stream_t stream);

/* Weight and bias gradients in one pass over g:  dw as conv_bwd_filter (bit for bit) and
 * db[oc] = sum over b, oh, ow of g (as conv_bwd_bias, up to summation order).  On the
 * tensor-core path the bias gradient is fused into wgrad: the threads that load and mask g
 * for the first k-tile of each split also sum it per output channel (each thread its
 * channel's values, chunk by chunk, in ascending column order), write one fp32 partial per
 * (split, lane group) after the split-K partials in the workspace, and the split reduction
 * adds them in ascending order -- so dy and y are read once for both gradients.  The other
 * families run the bias-gradient kernel after the weight gradient.
 *   x, dy, y, dw, workspace, workspace_bytes: as conv_bwd_filter (the same workspace size,
 *   conv_bwd_filter_workspace_size, serves both)   db: (OC), written. */
int conv_bwd_filter_bias(const conv_desc_t* desc, const void* x, const void* dy, const void* y, void* dw,
                         void* db, void* workspace, size_t workspace_bytes, conv_stream_t stream);

/* The whole backward in one call:  dx as conv_bwd_data, dw as conv_bwd_filter and, when db is
 * not NULL, db as conv_bwd_filter_bias -- PufferLib PR #522 times "backward" as wgrad plus
 * d_input together.  On the tensor-core path, while d_input's own launch would have fewer than
 * two waves of work items (the encoder layers up to a few thousand samples), d_input and wgrad
 * run in ONE launch (after W^T is packed into the workspace, and before the split reduction), one
 * work item per CTA: first the wgrad tiles (the long items), then d_input's work items cut into
 * k-tile ranges (short items: disjoint dx channels, no reduction), so that d_input fills the SMs
 * the wgrad tiles leave idle and backfills the others as they finish.  Each operation computes
 * exactly as in its own kernel, but wgrad splits the batch into fewer ranges than
 * conv_bwd_filter (its tiles then fill about two thirds of the SMs), so dw may differ from
 * conv_bwd_filter's in the last bits (same tolerance, deterministic); dx is bit for bit
 * conv_bwd_data's.  Otherwise
 * (conv_query(CONV_OP_BWD) reports algo CONV_ALGO_AUTO) conv_bwd_data's workspace path and
 * conv_bwd_filter run one after the other, each with its own part of the workspace.
 *   x, dy, w, y (required when relu): inputs; dx, dw, db (may be NULL): written.
 *   workspace: at least conv_bwd_workspace_size(desc) bytes, 16-byte aligned, owned by the
 *   caller, contents ignored on entry and unspecified on return. */
size_t conv_bwd_workspace_size(const conv_desc_t* desc);
int conv_bwd(const conv_desc_t* desc, const void* x, const void* dy, const void* w, const void* y, void* dx,
             void* dw, void* db, void* workspace, size_t workspace_bytes, conv_stream_t stream);

/* Bias gradient:  db[oc] = sum over b, oh, ow of g (g = dy masked by y > 0 when
 * relu), accumulated in fp32 and rounded once to the dtype.  One kernel: the
 * channels are cut into windows and the batch into R contiguous sample ranges
 * (R a power of two, at most 8); the CTA of (window, range) sums each output
 * position (oc, oh, ow) of its window down its rows (in interleaved row lanes,
 * each in ascending b), then adds, per channel, its positions in ascending
 * (oh, ow), each over the row lanes in ascending order; the R CTAs of a window
 * form a thread-block cluster whose rank-0 CTA adds the R per-channel sums in
 * ascending range order through distributed shared memory.  No global scratch.
 * A shape whose OH*OW is longer than 12288 positions runs a one-warp-per-channel
 * kernel instead (the same result up to summation order).
 *   dy: (B,OC,OH,OW)  y: forward output, required when desc->relu, ignored
 *   otherwise (may be NULL)  db: (OC), written (zeros when B = 0).
 * conv_query(CONV_OP_BWD_BIAS, ...) reports the plan (splits = R); conv_set_algo accepts
 * CONV_ALGO_AUTO and CONV_ALGO_DIRECT (the one-warp-per-channel kernel) for it. */
int conv_bwd_bias(const conv_desc_t* desc, const void* dy, const void* y, void* db,
                  conv_stream_t stream);

/* Two-layer forward chain:  y1 = act1(conv1(x, w1) + bias1),  y2 = act2(conv2(y1, w2) + bias2),
 * where layer 2's input is layer 1's output (d2->IC = d1->OC, d2->H x d2->W = layer 1's
 * OH x OW, same B and dtype) -- the encoder of PufferLib PR #522, whose layer-1 (11x15, K=5,
 * S=3, ReLU -> 3x4) and layer-2 (3x4, K=3, S=1 -> 1x2) bench blocks are its two halves.  act1 /
 * act2 follow d1->relu / d2->relu; bias1 / bias2 may be NULL (no bias).  y1 is written too
 * (the backward needs it as a mask source and as layer 2's input).  Results: y1 as conv_fwd /
 * conv_fwd_bias on layer 1 and y2 as conv_fwd on y1 -- bit for bit where those calls sum K in
 * one range, else up to summation order (they split K when their column tiles are few).
 * On the tensor-core path one kernel computes both layers per group of whole samples: layer 1's
 * output tile goes to y1 and into shared memory, where layer 2 gathers its input from, so y1
 * makes no round trip through memory between the layers and layer 2 needs no launch of its
 * own; both weight images are packed into the workspace first (two small kernels).  The fused
 * kernel runs in bf16 when every CTA gets at most one group of whole samples (the encoder: B up
 * to about 1500 on 152 SMs).  In fp32 the two forward calls were measured faster, so it runs
 * there only when conv_set_algo(CONV_OP_FWD, CONV_ALGO_TC) forces it.  Larger batches, fp32
 * unforced, and shapes the fused kernel does not take (a layer with
 * more than 128 output positions, layer 1 with more output channels than one tensor-core tile --
 * 128 fp32 / 256 bf16 --, layer 2 with more than 128), run as two conv_fwd_ws calls sharing the
 * workspace.
 *   workspace: at least conv_fwd_chain2_workspace_size(d1, d2) bytes, 16-byte aligned, owned
 *   by the caller; contents ignored on entry and unspecified on return.
 * conv_query_chain2 reports the plan (algo CONV_ALGO_TC when fused, CONV_ALGO_AUTO when it runs
 * as two forward calls); conv_set_algo(CONV_OP_FWD, ...) other than AUTO / TC disables the
 * fused kernel (and forces that family for the two calls). */
size_t conv_fwd_chain2_workspace_size(const conv_desc_t* d1, const conv_desc_t* d2);
int conv_fwd_chain2(const conv_desc_t* d1, const conv_desc_t* d2, const void* x, const void* w1, const void* bias1,
                    const void* w2, const void* bias2, void* y1, void* y2, void* workspace, size_t workspace_bytes,
                    conv_stream_t stream);

/* Two-layer backward chain, the backward of conv_fwd_chain2's stack (d1, d2 as there):
 *   g2 = dy2 masked by y2 > 0 when d2->relu;  dx2 = conv_bwd_data(g2, w2);  dw2, db2 from g2;
 *   g1 = dx2 masked by y1 > 0 when d1->relu;  dw1, db1 from g1;  dx1 = conv_bwd_data(g1, w1).
 * Layer 2 runs as conv_bwd (d_input and wgrad of the layer in one launch where that call fuses
 * them) with dx2 written into the workspace, not to a caller buffer: it is layer 1's dy and is
 * read back at once (6.3 MB in fp32 at the encoder's B = 1024, so it stays in L2).  Layer 1
 * runs as conv_bwd when dx1 is wanted, else as conv_bwd_filter / conv_bwd_filter_bias only --
 * the input gradient of a network's first layer is not needed.  Layer 1's wgrad reduces g1
 * over the whole batch, so dx2 has to be complete before it starts: the two layers are two
 * fused calls, one after the other on the stream, not one kernel.  Results as those calls.
 *   x1: layer 1's input  w1, w2: weights  y1: layer 1's output (layer 2's input and layer 1's
 *   mask source; required)  y2: layer 2's output (required when d2->relu, else may be NULL)
 *   dy2: (B, OC2, OH2, OW2)  dx1: NCHW like x1, or NULL (not computed)  dw1, dw2: written
 *   db1, db2: the bias gradients, or NULL (not computed).
 *   workspace: at least conv_bwd_chain2_workspace_size(d1, d2) bytes, 16-byte aligned, owned
 *   by the caller; contents ignored on entry and unspecified on return.
 * Errors: CONV_ERR_DESC when the descriptors do not chain (checked before any CUDA call), then
 * as conv_bwd. */
size_t conv_bwd_chain2_workspace_size(const conv_desc_t* d1, const conv_desc_t* d2);
int conv_bwd_chain2(const conv_desc_t* d1, const conv_desc_t* d2, const void* x1, const void* w1, const void* y1,
                    const void* w2, const void* y2, const void* dy2, void* dx1, void* dw1, void* db1, void* dw2,
                    void* db2, void* workspace, size_t workspace_bytes, conv_stream_t stream);

/* Weight gradient that allocates nothing (PufferLib PR #522 has no counterpart; this
 * entry point exists for callers of this library that cannot allocate device
 * memory: hosts that hand the library only the input and output buffers and own
 * every other byte, and code that must not allocate while a step runs, where an
 * allocation can block on the device or fail under memory pressure).
 *
 * Computes the same dw as conv_bwd_filter with the same split-K FFMA kernels,
 * but the fp32 split-K partials live in a scratch array inside the library: a
 * file-scope __device__ array of CONV_NOALLOC_SCRATCH_BYTES that every GPU which
 * loads the library holds until the process exits.  The number of split-K
 * ranges is capped so the partials fit; a descriptor whose single partial
 * (OC * round_up(IC*K*K, 4) * 4 bytes) exceeds the array is rejected with
 * CONV_ERR_UNSUPPORTED before anything is enqueued.  No workspace is passed and
 * the call makes no cudaMalloc / cudaFree and no allocating library call.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array: calls that overlap on the GPU
 * (e.g. on two streams, or from two threads) race and corrupt each other's
 * result.  Nothing in the array needs to start at zero: every partial the
 * reduction reads is written first by the same call.
 *   x, dy, y, dw, stream: as for conv_bwd_filter. */
#define CONV_NOALLOC_SCRATCH_BYTES (16u << 20)
int conv_bwd_filter_noalloc(const conv_desc_t* desc, const void* x, const void* dy, const void* y,
                            void* dw, conv_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* conv_status_string(int status);

/* Output spatial size for a descriptor (host-only validation helper). */
int conv_out_dims(const conv_desc_t* desc, int32_t* OH, int32_t* OW);

/* Launch plan for one operation on the current device, as the next call
 * with this descriptor would run it. */
typedef struct {
    int32_t algo;         /* conv_algo_t actually used                        */
    int32_t launches;     /* kernels enqueued per call                        */
    int32_t grid;         /* CTAs of the main kernel                          */
    int32_t block;        /* threads per CTA of the main kernel               */
    int32_t smem_bytes;   /* dynamic shared memory of the main kernel         */
    int32_t splits;       /* wgrad: number of split-K ranges (else 0)         */
    size_t workspace;     /* wgrad: workspace bytes (else 0)                  */
} conv_plan_info_t;
int conv_query(int op, const conv_desc_t* desc, conv_plan_info_t* info);
/* The plan of conv_fwd_chain2 for these two descriptors (see there). */
int conv_query_chain2(const conv_desc_t* d1, const conv_desc_t* d2, conv_plan_info_t* info);

/* The same plan for a device described by its properties instead of the current one,
 * computed on the host with no CUDA call (capacity planning; tests without a GPU).
 * sms: streaming multiprocessors; smem_optin: opt-in dynamic shared memory per block in
 * bytes; cc_major / cc_minor: compute capability (the tensor-core family needs
 * cc_major == 10).  The algorithm forced with conv_set_algo applies.  Returns
 * CONV_ERR_UNSUPPORTED for a property below 1 (cc_minor below 0). */
int conv_query_for_device(int op, const conv_desc_t* desc, int sms, int smem_optin, int cc_major, int cc_minor,
                          conv_plan_info_t* info);

/* Force an algorithm family for one operation (CONV_ALGO_AUTO restores the
 * library's choice).  Process-wide, not thread-safe; meant for tests and
 * benchmarks.  Returns CONV_ERR_UNSUPPORTED for an unknown op or algo, and for
 * CONV_ALGO_FFMA / CONV_ALGO_TC with CONV_OP_BWD_BIAS.  A forced family that
 * cannot run a given descriptor makes that call return CONV_ERR_UNSUPPORTED. */
int conv_set_algo(int op, int algo);

/* Diagnostics.  conv_fastdivmod_check runs, on the host, the library's
 * division-by-invariant-integer routine (Granlund & Montgomery, "Division by
 * invariant integers using multiplication", PLDI 1994) for divisor d over
 * every dividend in [lo, hi) and returns how many quotients or remainders
 * differ from '/' and '%'; (uint64_t)-1 if d is outside [1, 2^31). */
uint64_t conv_fastdivmod_check(uint32_t d, uint32_t lo, uint32_t hi);

/* Diagnostics: the tensor-core kernels bound every wait on an mbarrier; a wait
 * that runs out makes the kernel set a bit here, free its tensor memory and
 * return (its output is then unspecified).  Reads the word into *status
 * (0 = no timeout since the last reset), and clears it if reset != 0.
 * Synchronises the device. */
int conv_device_status(uint32_t* status, int reset);

/* Diagnostics: the timeout path of those waits, without a fault or a hang.  Enqueues on
 * `stream` one CTA whose thread waits on an mbarrier that nothing completes, through a
 * bounded loop of at most `max_sleeps` hardware sleeps of up to 1 microsecond each (the
 * kernels' own waits allow 4096 sleeps of up to 1 ms); when the loop runs out it sets bit 30
 * (CONV_STATUS_WAIT_SELFTEST) of the status word and returns normally, so the context stays
 * usable.  max_sleeps must be in [1, 10^6] (CONV_ERR_UNSUPPORTED otherwise). */
#define CONV_STATUS_WAIT_SELFTEST (1u << 30)
int conv_wait_selftest(uint32_t max_sleeps, conv_stream_t stream);

/* Write `bytes` bytes of `buf` (device memory, 16-byte aligned, bytes a
 * multiple of 16) on `stream`, evicting earlier data from L2; benchmarks use
 * it between timed iterations. */
int conv_l2_flush(void* buf, size_t bytes, conv_stream_t stream);

/* Library version, e.g. "0.1.0". */
const char* conv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* IGCONV_CONV_H */
