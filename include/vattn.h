/*
 * vattn.h -- C ABI of libvattn: non-causal multi-head attention over image
 * patches, head-major layout, on one NVIDIA GB300 (sm_103a) GPU.
 *
 * Operation (the shader "vision_attention_flash_sub_hpd_f16.wgsl",
 * rullama 0.1.0: its Params block, the head-major q/k/v/out buffers, the
 * tiled online-softmax loop over keys and the final o / l store):
 *
 *     out[b, h, i, :] = sum_j softmax_j( q[b,h,i,:] . k[b,h,j,:] ) * v[b,h,j,:]
 *
 * for every batch entry b, head h and patch (query) i, the softmax running
 * over all n_patches keys j of the same (b, h).  No 1/sqrt(head_dim) factor
 * is applied: the caller passes q already scaled.  Like the shader, the
 * kernel rounds q, k, v and the softmax weights to f16 for the two matrix
 * products and keeps the softmax statistics (running max m, running sum l)
 * and the accumulator o in f32.  The shader has no batch dimension; here
 * batch is folded into the head index (b * n_heads + h), which is exactly
 * how a contiguous [batch, n_heads, n_patches, head_dim] buffer is laid out.
 *
 * Threading: entry points are thread-safe; the last-error text is kept per
 * host thread.
 */
#ifndef VATTN_H_
#define VATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VATTN_OK = 0,
  VATTN_ERR_INVALID_ARG = 1,    /* negative size, null pointer, aliasing out */
  VATTN_ERR_UNSUPPORTED = 2,    /* head_dim > 128, sizes past 32-bit indexing */
  VATTN_ERR_MISALIGNED = 3,     /* pointer not aligned to its element (4 bytes) */
  VATTN_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  VATTN_ERR_DEVICE_TIMEOUT = 5  /* a kernel-side wait ran out (see vattn_device_status) */
} vattn_status;

/* Largest head_dim the kernel handles. */
#define VATTN_MAX_HEAD_DIM 128

/*
 * vattn_forward -- out = softmax(q k^T) v per (batch, head).
 *
 * q, k, v, out: DEVICE pointers (memory of the device current on the calling
 *   thread) to contiguous f32 tensors of shape
 *   [batch, n_heads, n_patches, head_dim], head-major: element (b, h, i, d)
 *   sits at ((b * n_heads + h) * n_patches + i) * head_dim + d.  q must be
 *   pre-scaled (typically by 1/sqrt(head_dim)).
 * out must not overlap q, k or v.  The caller owns all four buffers; the
 *   library keeps no reference to them after the call returns.
 * head_dim: 1..128.  Any n_patches >= 0 (ragged tails are handled).
 * stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *
 * The call is asynchronous: it validates arguments, launches its kernels on
 * `stream` and returns; the result is ready when the stream reaches that
 * point.  Three paths, the same f16 rounding and, for the same work
 * schedule, bit-identical results (where the last round of work tiles is
 * cut between blocks, see vattn_set_split_tiles, a row's last bits depend on
 * that schedule):
 *   - 128 < n_patches <= 1536 with head_dim 33..64, or up to 2048 patches
 *     while the work tiles (batch*n_heads * ceil(n_patches / 256)) fill at
 *     most two rounds of the multiprocessors, or n_patches <= 128 with
 *     head_dim <= 64; head_dim a multiple of 4, q, k, v 16-byte aligned:
 *     one kernel that reads the f32 tiles and rounds them to f16 in shared
 *     memory; nothing is allocated;
 *   - otherwise, with head_dim <= 64 and a multiple of 4 and q, k, v
 *     16-byte aligned and more than 128 patches: a memset and one
 *     cooperative kernel that writes the f16 copies of k and v itself,
 *     each key tile once, while its blocks compute (a block reads a key
 *     tile once the block that wrote it has set the tile's flag), and
 *     rounds q itself;
 *   - otherwise two kernels (the f16 staging of q, k and v, then the
 *     attention kernel; the attention kernel rounds q itself when head_dim
 *     <= 64 and q is 16-byte aligned, and the staging kernel then k and v
 *     only).
 *   The f16 copies and flags (at most 3 * batch*n_heads*n_patches*
 *   round_up(head_dim, 16) * 2 bytes) live in a workspace taken
 *   stream-ordered from a memory pool the library keeps per device
 *   (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`; the pool keeps
 *   its memory between calls).
 * batch*n_heads == 0 or n_patches == 0 is a successful no-op that launches
 * nothing.
 *
 * Returns VATTN_OK, or an error code with no kernel launched (argument
 * errors are detected on the host, before any CUDA call), or VATTN_ERR_CUDA
 * if the workspace allocation or a launch failed.  Errors raised while the kernel runs are
 * reported by vattn_device_status().
 */
vattn_status vattn_forward(const float* q, const float* k, const float* v, float* out,
                           int64_t batch, int64_t n_heads, int64_t n_patches,
                           int64_t head_dim, void* stream);

/*
 * vattn_forward_f16 -- the same attention on inputs that are already f16.
 *
 * The shader rounds q, k and v to f16 as it stages them in workgroup
 * storage (its q_shared / kv_tile declarations); vattn_forward does that
 * rounding in a first kernel.  Callers whose activations are already f16
 * skip it here: this call launches the attention kernel alone, which reads
 * the caller's tensors directly with TMA.  The result equals vattn_forward
 * on the f32 values of these f16 inputs (the same kernel, the same
 * arithmetic).
 *
 * q, k, v: DEVICE pointers to contiguous IEEE binary16 tensors (bit
 *   patterns as uint16_t) of shape [batch, n_heads, n_patches, head_dim],
 *   head-major, q pre-scaled; 16-byte aligned.
 * out: DEVICE pointer to f32 [batch, n_heads, n_patches, head_dim], 4-byte
 *   aligned, not overlapping q, k or v.  The caller owns all buffers.
 * head_dim: 8..128, a multiple of 8 (rows must span whole 16-byte units);
 *   other values return VATTN_ERR_UNSUPPORTED (use vattn_forward).
 * stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *
 * Asynchronous, no allocation, one kernel launch; empty problems are a
 * no-op.  Errors as for vattn_forward (argument errors on the host before
 * any CUDA call).
 */
vattn_status vattn_forward_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               float* out, int64_t batch, int64_t n_heads, int64_t n_patches,
                               int64_t head_dim, void* stream);

/*
 * vattn_forward_f16io -- vattn_forward_f16 with an f16 output: each output
 * element is the f32 value vattn_forward_f16 would store, rounded to f16
 * (round to nearest even).  Halves the output bytes for callers that keep
 * activations in f16.
 *
 * q, k, v: as for vattn_forward_f16 (f16, head_dim % 8 == 0, 16-byte
 *   aligned).  out: DEVICE pointer to IEEE binary16 [batch, n_heads,
 *   n_patches, head_dim], 2-byte aligned (16-byte aligned lets the kernel
 *   write it with bulk tensor stores), not overlapping q, k or v.
 * Asynchronous, no allocation, one kernel launch; errors as for
 * vattn_forward_f16.
 */
vattn_status vattn_forward_f16io(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* out, int64_t batch, int64_t n_heads,
                                 int64_t n_patches, int64_t head_dim, void* stream);

/*
 * vattn_forward_f32q -- attention with f32 queries and f16 keys and values.
 *
 * For callers that hold k and v in f16 (computed once, attended by fresh
 * f32 queries).  The kernel rounds q to f16 itself (round to nearest even)
 * once per block of query rows, so the result equals vattn_forward on q and
 * the f32 values of k and v, bit for bit.
 *
 * q, out: DEVICE f32 [batch, n_heads, n_patches, head_dim]; k, v: DEVICE
 *   IEEE binary16 tensors of the same shape.  q, k, v 16-byte aligned, out
 *   4-byte aligned, out not overlapping q, k or v.
 * Shapes: head_dim a multiple of 8 and at most 64, n_patches > 128 (the
 *   kernel variant with two 128-row query tiles per block); other shapes
 *   return VATTN_ERR_UNSUPPORTED (round q to f16 and call vattn_forward_f16).
 * Asynchronous, no allocation, one kernel launch; errors as for
 * vattn_forward_f16.
 */
vattn_status vattn_forward_f32q(const float* q, const uint16_t* k, const uint16_t* v, float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, void* stream);

/*
 * vattn_rope_neox -- NeoX rotary position embedding, in place.
 *
 * The rotation of the WGSL kernel "rope_neox_backward.wgsl" (rullama 0.2.0):
 * with half = rope_dims / 2, in every row the pair (x[i], x[i + half]),
 * i < half, is turned by theta_i = pos * base^(-2 i / rope_dims), divided by
 * factors[i] when factors is not NULL:
 *   inverse == 0 (forward): x[i] <- a cos - b sin,  x[i + half] <- a sin + b cos
 *   inverse == 1 (backward): x[i] <- a cos + b sin, x[i + half] <- -a sin + b cos
 * with a = x[i], b = x[i + half]; dims >= 2 * half are not touched.  theta,
 * cos and sin are computed in f32 as on the page (f32(pos) * pow(base,
 * -2 i / rope_dims), then / factors[i]).
 *
 * x: DEVICE pointer to a contiguous f32 tensor [batch, n_heads, n_patches,
 *   head_dim] (head-major, 4-byte aligned); patch n is at position
 *   pos0 + n.  (With n_patches == 1 and pos0 == pos this is the page's
 *   kernel on [n_heads, head_dim].)
 * rope_dims: 0..head_dim (odd values leave dim rope_dims - 1 alone, as the
 *   page's integer half does); base: finite, > 0; pos0 >= 0 with
 *   pos0 + n_patches <= 2^24 (positions exact in f32); factors: NULL or a
 *   DEVICE pointer to rope_dims / 2 floats.
 * Asynchronous on `stream`; a small angle table (n_patches * rope_dims / 2
 * * 8 bytes) is taken stream-ordered from the library's memory pool.
 * Argument errors are returned before any CUDA call.
 */
vattn_status vattn_rope_neox(float* x, int64_t batch, int64_t n_heads, int64_t n_patches,
                             int64_t head_dim, int64_t rope_dims, int64_t pos0, float base,
                             const float* factors, int inverse, void* stream);

/*
 * vattn_forward_rope -- vattn_forward on q and k turned by the forward NeoX
 * rotation of vattn_rope_neox (patch n at position pos0 + n), fused into the
 * f16 staging pass: q and k are read once, rotated in f32 and rounded to f16;
 * the caller's q and k are not modified.  The rotation is the one the page
 * "rope_neox_backward.wgsl" applies around attention; the attention is that
 * of vattn_forward.  Arguments and errors: those of vattn_forward and of
 * vattn_rope_neox.  Workspace: vattn_forward's plus the angle table.
 */
vattn_status vattn_forward_rope(const float* q, const float* k, const float* v, float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, int64_t rope_dims, int64_t pos0, float base,
                                const float* factors, void* stream);

/*
 * vattn_forward_accurate -- the attention of vattn_forward without the f16
 * rounding of the operands, to about f32 accuracy.
 *
 * The shader's header comment names a sibling variant, "sub", that keeps
 * q, k, v and the tile scores in f32 workgroup storage instead of f16; this
 * call is its counterpart.  It keeps the tensor cores by splitting every
 * operand in two f16 terms, x = hi + lo with hi = f16(x) and
 * lo = f16(x - hi) (round to nearest even), which represents x to about
 * 2^-22 relative, and takes three products for each of the two matrix
 * products:  S = Qh Kh^T + Qh Kl^T + Ql Kh^T  and, with the softmax weights
 * split the same way,  O += Ph Vh + Ph Vl + Pl Vh  (the dropped lo x lo
 * terms are below 2^-22 relative), all accumulated in f32.  Statistics,
 * accumulator and output are f32 as in vattn_forward.  It costs about three
 * times the tensor work of vattn_forward and twice its staged bytes.
 *
 * Arguments, layout, ownership and error codes: those of vattn_forward.
 * Workspace: six f16 tensors (hi and lo of q, k, v), 2 x vattn_forward's,
 * from the same per-device pool, stream-ordered.  Asynchronous; two kernel
 * launches; empty problems are a no-op.
 */
vattn_status vattn_forward_accurate(const float* q, const float* k, const float* v, float* out,
                                    int64_t batch, int64_t n_heads, int64_t n_patches,
                                    int64_t head_dim, void* stream);

/*
 * vattn_conv1d_step -- one step of a depthwise (per-channel) causal conv1d
 * whose past inputs live in a rolling buffer, for a batch of independent
 * sequences: the WGSL kernel "conv1d.wgsl" (cera 0.2.0), its header comment
 * and bindings.  For every sequence b and channel ch:
 *
 *   output[b, ch] = sum_{k < d_conv} buffer[b, k, ch] * weight[ch, k]
 *                   + input[b, ch] * weight[ch, d_conv]
 *
 * in f32, taps in that order, each product-and-add one fused multiply-add;
 * then, in place, buffer[b, k, ch] <- buffer[b, k + 1, ch] for
 * k < d_conv - 1 and buffer[b, d_conv - 1, ch] <- input[b, ch] (slot 0 is
 * the oldest).  With batch == 1 this is exactly the page's kernel.
 *
 * input, output: DEVICE pointers to f32 [batch, hidden_size].
 * buffer: DEVICE pointer to f32 [batch, d_conv, hidden_size] (each
 *   sequence's block is the page's [d_conv, hidden_size] layout, slot k of
 *   channel ch at k * hidden_size + ch), read and rewritten; may be NULL
 *   when d_conv == 0.
 * weight: DEVICE pointer to f32 [hidden_size, kernel_size], tap k of
 *   channel ch at ch * kernel_size + k, shared by all sequences; taps past
 *   d_conv are not read.  kernel_size >= d_conv + 1.
 * All 4-byte aligned (hidden_size % 4 == 0, d_conv <= 8 and 16-byte aligned
 * input, buffer and output take 16-byte accesses).  output must not overlap
 * input, buffer or weight; buffer must not overlap input or weight.  The
 * caller owns all buffers.
 *
 * Asynchronous on `stream`, one kernel launch, no allocation; batch == 0 or
 * hidden_size == 0 is a no-op.  Calls that update one buffer must be
 * ordered (one stream, or events).  Argument errors are returned before any
 * CUDA call: VATTN_ERR_INVALID_ARG (negative size, kernel_size < d_conv + 1,
 * null pointer, overlap), VATTN_ERR_UNSUPPORTED (sizes past 32 bits or byte
 * sizes past 64), VATTN_ERR_MISALIGNED; VATTN_ERR_CUDA if the launch fails.
 */
vattn_status vattn_conv1d_step(const float* input, float* buffer, const float* weight,
                               float* output, int64_t batch, int64_t hidden_size,
                               int64_t kernel_size, int64_t d_conv, void* stream);

/*
 * vattn_forward_host -- vattn_forward on HOST buffers: q, k, v are read from
 * host memory and out is written to host memory, with the copies pipelined
 * against the kernels.
 *
 * The heads (batch * n_heads) are cut into up to eight chunks of whole heads.
 * Three streams the library keeps per device carry, for each chunk, the
 * host-to-device copies of its q, k and v, the kernels of vattn_forward (the
 * direct f32 kernel, else the staging kernel and the attention kernel: not
 * the single cooperative kernel), and the device-to-host copy of its output,
 * so that the copies of one chunk overlap the kernels of the next.  Tiles
 * are never cut here, so the result is bit-identical to vattn_forward on
 * the same values with cutting forbidden (vattn_set_split_tiles(0)); with
 * the default setting, to within the rounding of the cut tiles' merge.
 *
 * q, k, v, out: HOST pointers to contiguous f32 [batch, n_heads, n_patches,
 *   head_dim], head-major, 4-byte aligned; out must not overlap q, k or v.
 *   Page-locked memory (cudaHostAlloc / cudaHostRegister) lets the copies
 *   run asynchronously and overlap; pageable memory gives the same result
 *   with the copies serialised by the driver.
 * stream: a cudaStream_t passed as void* (NULL = legacy default stream).  The
 *   work is ordered after what was queued on `stream` and `stream` continues
 *   only after the last copy out: out may be read once `stream` has been
 *   synchronised.  The caller must keep all four buffers alive until then.
 * Workspace (stream-ordered on `stream`, from the library's per-device pool):
 *   two chunks of f32 inputs and outputs plus one chunk of f16 staging.
 * Errors: those of vattn_forward; argument errors on the host before any
 *   CUDA call.
 */
vattn_status vattn_forward_host(const float* q, const float* k, const float* v, float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, void* stream);

/*
 * Size of the fixed staging scratch of vattn_forward_noalloc: 32 MiB, enough
 * for batch*n_heads*n_patches*round_up(head_dim, 16) <= 5,592,320 (for
 * example 16 heads x 4,100 patches at head_dim 72, or 64 heads x 1,024
 * patches at head_dim 64).
 */
#define VATTN_NOALLOC_MAX_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * Size of the second fixed array of vattn_forward_noalloc: the flags a call
 * clears at its start and the partial results of tiles that the work
 * schedule cuts between two thread blocks (16 MiB: room for every schedule
 * on a GPU of up to 152 multiprocessors).
 */
#define VATTN_NOALLOC_PART_BYTES (16u * 1024u * 1024u)

/*
 * vattn_forward_noalloc -- vattn_forward without any device memory
 * allocation.  The shader this library follows has no counterpart: it is an
 * interface for callers that may not allocate while they run, such as a
 * plugin inside an inference runtime that owns all device memory and forbids
 * allocation in its execute step, or a latency-bound loop that cannot take an
 * allocation's cost or a late out-of-memory failure.
 *
 * Arguments, layout, result and error codes are those of vattn_forward, and
 * so are its kernels and its mode (vattn_forward_mode).  The workspace that
 * vattn_forward takes from its pool goes to a fixed array of
 * VATTN_NOALLOC_MAX_SCRATCH_BYTES that the library's device code holds on
 * every device it is loaded on (for the life of the process): the f16
 * copies of q, k and v in the two-kernel mode; the f16 copies of k and v,
 * written by the attention kernel itself, and one ready flag per (head, key
 * tile) in the single cooperative kernel's mode.  The call makes no
 * cudaMalloc/cudaFree-type call; the flags are cleared by a memset on
 * `stream` at the start of each call.
 *
 * Limit: a problem whose f16 copies (3 x 256-byte-rounded
 * batch*n_heads*n_patches*round_up(head_dim, 16)*2 bytes) exceed the array is
 * rejected on the host with VATTN_ERR_UNSUPPORTED and nothing launched; use
 * vattn_forward for it.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call outside any stream capture.
 *
 * Calls that can overlap in time on one device -- on different streams, or
 * from several host threads -- share the one array and race, on the f16
 * copies and on the ready flags: their results are undefined (a flag that
 * another call clears can also make a wait run out, which ends in
 * VATTN_ERR_DEVICE_TIMEOUT from vattn_device_status, not in a hang).
 * Order them (one stream, or events) or use vattn_forward.  Apart from the
 * flags, which each call clears, nothing in the array needs to start at
 * zero: each call writes what it reads.
 */
vattn_status vattn_forward_noalloc(const float* q, const float* k, const float* v, float* out,
                                   int64_t batch, int64_t n_heads, int64_t n_patches,
                                   int64_t head_dim, void* stream);

/*
 * Kernel modes of vattn_forward (all give bit-identical results for the
 * same work schedule: the same f16 rounding and the same tensor-core
 * arithmetic).  The shader has one
 * compute pass per call; these are this library's ways of scheduling it.
 *   VATTN_MODE_NONE           empty problem: nothing is launched;
 *   VATTN_MODE_DIRECT         one kernel on the f32 tiles (q, k, v rounded
 *                             to f16 in shared memory), no workspace;
 *   VATTN_MODE_SINGLE_KERNEL  a memset of key-tile flags and one cooperative
 *                             kernel that writes the f16 copies of k and v
 *                             itself while it computes;
 *   VATTN_MODE_TWO_KERNELS    the f16 staging kernel, then the attention
 *                             kernel.
 */
typedef enum {
  VATTN_MODE_NONE = 0,
  VATTN_MODE_DIRECT = 1,
  VATTN_MODE_SINGLE_KERNEL = 2,
  VATTN_MODE_TWO_KERNELS = 3
} vattn_mode;

/*
 * vattn_forward_mode -- the mode (vattn_mode) that vattn_forward takes, on
 * the current device, for exactly these arguments.  Checks the arguments
 * as vattn_forward does (same error codes, on the host) and launches
 * nothing.  The first query on a device that could take the single
 * cooperative kernel reads the device's cooperative-launch support and the
 * kernel's occupancy (CUDA calls; cached per device).  vattn_forward_noalloc
 * takes the same mode; vattn_forward_host never takes the single kernel.
 * The shader has no counterpart: this exists for callers that plan memory
 * or launches, and for tests.
 */
vattn_status vattn_forward_mode(const float* q, const float* k, const float* v, const float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, int* mode);

/*
 * vattn_forward_mode_for -- the rule behind vattn_forward_mode, with the
 * device facts passed in instead of read from a device: aligned = q, k and
 * v are all 16-byte aligned; cooperative_launch = the device attribute
 * cudaDevAttrCooperativeLaunch; blocks_per_sm = resident blocks per
 * multiprocessor of the single cooperative kernel (0 when it does not fit);
 * n_sms = the device's multiprocessors (>= 1; VATTN_ERR_INVALID_ARG
 * otherwise), the size of the persistent grid.  The single kernel is taken
 * only when cooperative_launch != 0, blocks_per_sm >= 1 and
 * vattn_set_single_kernel has not forbidden it.  Pure host function (no
 * CUDA call).  Sizes are checked as in vattn_forward; *mode =
 * VATTN_MODE_NONE for an empty problem.
 */
vattn_status vattn_forward_mode_for(int64_t batch, int64_t n_heads, int64_t n_patches,
                                    int64_t head_dim, int aligned, int cooperative_launch,
                                    int blocks_per_sm, int n_sms, int* mode);

/*
 * vattn_set_single_kernel -- allow (allow != 0, the default) or forbid
 * (allow == 0) the single cooperative kernel, process-wide.  Forbidden, the
 * calls that would take it take VATTN_MODE_TWO_KERNELS instead (same
 * result, one more kernel); useful where cooperative grids are not wanted,
 * for example on a GPU shared under MPS with a limit on multiprocessors.
 * (Without the switch, a cooperative launch that the driver refuses as too
 * large also falls back to the two kernels.)  Returns the previous setting
 * (1 or 0).  Not synchronised with calls in flight on other host threads:
 * set it before them.
 */
int vattn_set_single_kernel(int allow);

/*
 * vattn_set_split_tiles -- cut work tiles where it pays (allow == 1, the
 * default), never (allow <= 0), or wherever it shortens the busiest block
 * (allow >= 2, for tests and measurements), process-wide.  The attention kernel is
 * persistent (one thread block per multiprocessor); when the work tiles
 * (128 or 256 query rows of one head) do not divide evenly over the blocks,
 * vattn_forward and vattn_forward_noalloc may cut the tiles of the last
 * round(s) by key range, one equal share per block, and the two parts of a
 * cut tile are combined by the log-sum-exp rule (the shader's rescale of
 * (m, l, o)).  They do so only where it pays, measured on GB300: tiles of at
 * least 16 key tiles (2048 patches) and a busiest block shorter by at least
 * 7 key tiles (for example 8 x 16 heads x 2304 patches, or 2 x 16 heads x
 * 4096 patches, 8 % faster).  The result is the same attention, but the
 * rounding of a cut tile's rows then depends on how the call's work was
 * shared out, i.e. on the other heads in the call.  Forbidden, every tile
 * runs whole in one block: each output row depends only on its own head's
 * inputs (bit-identical whatever else the call holds, as in
 * vattn_forward_f16 / _f32q / _host, which never cut), at the price of a
 * partial last round.  Not synchronised with calls in flight on other host
 * threads: set it before them.  The shader
 * has no counterpart (one workgroup per block of rows).  Returns the
 * previous setting (0, 1 or 2).
 */
int vattn_set_split_tiles(int allow);

/*
 * vattn_cut_plan_for -- host-only query: whether vattn_forward would cut
 * work tiles (see vattn_set_split_tiles) for q, k, v of these sizes on a
 * device whose persistent grid has n_blocks thread blocks (its
 * multiprocessor count), under the current process-wide setting.  *cut: 1
 * or 0 (0 for an empty problem).  No GPU is touched.  Errors: a null `cut`,
 * n_blocks < 1 or sizes outside the limits of vattn_forward (the same
 * status as vattn_forward for those).  The shader has no counterpart.
 */
vattn_status vattn_cut_plan_for(int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, int n_blocks, int* cut);

/*
 * vattn_device_status -- reads and clears the kernel-side error word of the
 * current device.  Every wait inside the kernel is bounded; one that runs
 * out sets a non-zero code (which wait, in the low byte) and the thread
 * block ends early with its output rows unwritten.  Synchronises the
 * current device first.  *code receives 0 when no kernel failed.
 * Returns VATTN_OK, VATTN_ERR_DEVICE_TIMEOUT if *code != 0, or
 * VATTN_ERR_CUDA / VATTN_ERR_INVALID_ARG.
 */
vattn_status vattn_device_status(uint32_t* code);

/*
 * vattn_selftest_wait_timeout -- exercises the kernels' failure detection
 * without faulting anything: launches on `stream` a one-thread kernel whose
 * bounded wait, the same as every wait in the attention kernel, is on an
 * mbarrier phase that nothing completes.  After the wait limit (about 2 s)
 * it records a timeout with site code 15 in the status word and returns;
 * the device stays usable.  vattn_device_status() then returns
 * VATTN_ERR_DEVICE_TIMEOUT with *code == 0x10F and clears the word.  The
 * shader has no counterpart: this exists to test the timeout path.
 * Returns VATTN_OK once launched, or VATTN_ERR_CUDA.
 */
vattn_status vattn_selftest_wait_timeout(void* stream);

/* Static text for a status code. */
const char* vattn_status_string(vattn_status status);

/* Detail text of the last error on this host thread ("" if none). */
const char* vattn_last_error_string(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int vattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VATTN_H_ */
