// vattn_api.cu -- the C ABI declared in include/vattn.h: argument checks,
// workspace, tensor-map encoding, variant choice and the two launches of a
// call (f16 staging of q/k/v, then the attention kernel) on sm_103a.
//
// The operation is the one of the WGSL shader
// "vision_attention_flash_sub_hpd_f16.wgsl" (rullama 0.1.0): its Params block
// (head_dim, n_heads, n_patches) becomes plain integer arguments plus a
// batch size folded into the head index; its four storage buffers become
// device pointers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/vattn.h"
#include "attn_kernel.cuh"
#include "conv1d_kernel.cuh"
#include "rope_kernel.cuh"
#include "stage_kernel.cuh"

namespace {

thread_local char g_last_error[512] = "";

vattn_status fail(vattn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

vattn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(VATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// cuTensorMapEncodeTiled, fetched from the driver at run time so that the
// library itself does not link against libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// 3-D view {cols, n_patches, batch*n_heads} of a head-major f16 tensor whose
// rows hold `cols` elements; one box = 128 rows x 64 columns (128 bytes),
// 128-byte swizzle: the layout the tensor-core descriptors expect.
// Out-of-range rows and columns read 0.  cols * 2 must be a multiple of 16.
vattn_status make_tmap16(CUtensorMap* tm, const __half* ptr, int64_t bh, int64_t n, int cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    if (g_encode_err != cudaSuccess) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled lookup");
    return fail(VATTN_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(n),
                              static_cast<cuuint64_t>(bh)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2u,
                                 static_cast<cuuint64_t>(n) * static_cast<cuuint64_t>(cols) * 2u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(vattn::kBN), 1u};
  const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(ptr), dims,
                         strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(VATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult %d", static_cast<int>(r));
  return VATTN_OK;
}

// 3-D view {head_dim, n_patches, batch*n_heads} of the output for the
// kernel's TMA stores: box = 32 rows x 16 columns, f32 (64 bytes, 64-byte
// swizzle) or f16 (32 bytes, 32-byte swizzle): the layouts the kernel writes
// to its staging buffers.  Needs rows of whole 16-byte units (head_dim % 4 ==
// 0 for f32, % 8 == 0 for f16) and a 16-byte aligned base.
// f32 [bh, n, d] (d % 4 == 0, 16-byte aligned base) with boxes of {64
// columns, 128 rows}, no swizzle; columns past d and rows past n read as zero.
vattn_status make_tmap32(CUtensorMap* tm, const float* ptr, int64_t bh, int64_t n, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    if (g_encode_err != cudaSuccess) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled lookup");
    return fail(VATTN_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n),
                              static_cast<cuuint64_t>(bh)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4u,
                                 static_cast<cuuint64_t>(n) * static_cast<cuuint64_t>(d) * 4u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(vattn::kBM), 1u};
  const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims,
                         strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(VATTN_ERR_CUDA, "cuTensorMapEncodeTiled (f32) failed with CUresult %d", static_cast<int>(r));
  return VATTN_OK;
}

vattn_status make_tmap_out(CUtensorMap* tm, void* out, int64_t bh, int64_t n, int d, bool f16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    if (g_encode_err != cudaSuccess) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled lookup");
    return fail(VATTN_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n),
                              static_cast<cuuint64_t>(bh)};
  const cuuint64_t esize = f16 ? 2u : 4u;
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esize,
                                 static_cast<cuuint64_t>(n) * static_cast<cuuint64_t>(d) * esize};
  const cuuint32_t box[3] = {16u, 32u, 1u};
  const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
  const CUresult r = enc(tm, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         3, out, dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         f16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(VATTN_ERR_CUDA, "cuTensorMapEncodeTiled (out) failed with CUresult %d", static_cast<int>(r));
  return VATTN_OK;
}

constexpr int kMaxDevices = 64;

// Per-device memory pool for the f16 staging workspace: stream-ordered
// allocations, memory kept in the pool between calls.
struct DevicePool {
  std::once_flag once;
  cudaMemPool_t pool = nullptr;
  cudaError_t err = cudaSuccess;
};
DevicePool g_pools[kMaxDevices];

vattn_status pool_for(int device, cudaMemPool_t* out) {
  if (device < 0 || device >= kMaxDevices) return fail(VATTN_ERR_CUDA, "device index %d out of range", device);
  DevicePool& dp = g_pools[device];
  std::call_once(dp.once, [&dp, device] {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    dp.err = cudaMemPoolCreate(&dp.pool, &props);
    if (dp.err == cudaSuccess) {
      uint64_t keep = UINT64_MAX;
      dp.err = cudaMemPoolSetAttribute(dp.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
  });
  if (dp.err != cudaSuccess) return cuda_fail(dp.err, "creating the workspace memory pool");
  *out = dp.pool;
  return VATTN_OK;
}

// Streaming multiprocessors of a device, looked up once per device.
std::atomic<int> g_sm_count[kMaxDevices];

vattn_status sm_count(int device, int* out) {
  if (device < 0 || device >= kMaxDevices) return fail(VATTN_ERR_CUDA, "device index %d out of range", device);
  int n = g_sm_count[device].load(std::memory_order_acquire);
  if (n <= 0) {
    const cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessor count)");
    if (n <= 0) return fail(VATTN_ERR_CUDA, "device reports %d multiprocessors", n);
    g_sm_count[device].store(n, std::memory_order_release);
  }
  *out = n;
  return VATTN_OK;
}

// Work schedule of the persistent attention kernel over n_tiles tiles of T
// key tiles on `grid` blocks (the kernel's Sched).  Whole tiles in rounds;
// when the rounds leave a last, partial round (n_tiles % grid != 0) and
// cutting is allowed, the last one or two rounds' tiles are instead cut by
// key ranges into one equal share per block -- provided the tiles are long
// (at least kCutMinKeyTiles key tiles) and the cut shortens the busiest
// block by at least kCutMinSaving key tiles.  The pieces' extra prologues
// and the merges of the cut tiles cost, measured on GB300, the time of 5 to
// 10 key tiles per call (8 x 16 heads: +22 % at 1024 patches, tiles of 8 key
// tiles, saving 2; +2 % at 16 x 4100, saving 6; -1.3 % at 2304 patches,
// saving 7; 2 x 16 heads at 4096 patches: -8.2 %, saving 20).  Each share
// holds at least T key tiles (the tail has at least `grid` tiles), so a tile
// is cut at most once.
constexpr int kCutMinKeyTiles = 16;
constexpr int kCutMinSaving = 7;
struct Schedule {
  int rounds = 0;
  int extra = 0;
  long long tail_units = 0;
  bool cut = false;
};

// Process-wide switch of vattn_set_split_tiles: 0 never cut, 1 cut where it
// pays (the default), 2 cut wherever it shortens the busiest block.
std::atomic<int> g_cut_allowed{1};

Schedule make_schedule(long long n_tiles, int T, int grid, int cut_mode) {
  Schedule s;
  s.rounds = static_cast<int>(n_tiles / grid);
  s.extra = static_cast<int>(n_tiles % grid);
  if (cut_mode == 0 || s.extra == 0 || grid < 2) return s;
  const int r = n_tiles >= 2LL * grid ? s.rounds - 1 : 0;
  const long long tail = (n_tiles - static_cast<long long>(r) * grid) * T;
  const long long busiest_cut = static_cast<long long>(r) * T + (tail + grid - 1) / grid;
  const long long busiest_whole = static_cast<long long>(s.rounds + 1) * T;
  if (cut_mode == 1 && (T < kCutMinKeyTiles || busiest_cut + kCutMinSaving > busiest_whole)) return s;
  if (busiest_cut + 2 > busiest_whole) return s;
  s.rounds = r;
  s.extra = 0;
  s.tail_units = tail;
  s.cut = true;
  return s;
}

// f32 words of one partial slot (a cut tile's O, m, l for its nq query tiles)
size_t part_slot_floats(int nq, int d_pad) {
  return static_cast<size_t>(nq) * vattn::kBM * static_cast<size_t>(d_pad + 2);
}

// The attention kernel is persistent: one block per multiprocessor (at most
// one per tile), each looping over its share of the work (make_schedule).
// tql, tkl, tvl: the lo halves of q, k, v (accurate mode only; otherwise
// unused and any valid map may be passed).
template <int NQ, int NKB, bool kOut16, bool kAcc, int kIn = vattn::kInF16>
vattn_status launch_attention_maps(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tql,
                                   const CUtensorMap& tkl, const CUtensorMap& tvl,
                                   vattn::Params p, unsigned n_tiles, cudaStream_t stream,
                                   int device, bool* coop_refused = nullptr) {
  using P = vattn::Plan<NQ, NKB, kAcc, kIn>;
  auto kernel = vattn::vattn_fwd_kernel<NQ, NKB, kOut16, kAcc, kIn>;
  static std::atomic<uint8_t> configured[kMaxDevices];
  if (!configured[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         P::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    configured[device].store(1, std::memory_order_release);
  }
  int sms = 0;
  const vattn_status st = sm_count(device, &sms);
  if (st != VATTN_OK) return st;
  const unsigned grid = n_tiles < static_cast<unsigned>(sms) ? n_tiles : static_cast<unsigned>(sms);
  if (p.rounds == 0 && p.extra == 0 && p.tail_units == 0) {
    // no schedule given: whole tiles, round robin over the blocks
    p.rounds = static_cast<int>(n_tiles / grid);
    p.extra = static_cast<int>(n_tiles % grid);
  }
  // the output goes through TMA stores when the kernel variant stages it
  // (head_dim <= 64) and its rows are whole 16-byte units
  CUtensorMap to;
  std::memset(&to, 0, sizeof(to));
  p.tma_out = 0;
  if (P::kEpiBytes > 0 && p.vec_out) {
    void* out_base = kOut16 ? static_cast<void*>(p.out16) : static_cast<void*>(p.out);
    const vattn_status so = make_tmap_out(&to, out_base, static_cast<int64_t>(p.n_tiles / p.n_qblocks),
                                          p.n_patches, p.head_dim, kOut16);
    if (so != VATTN_OK) return so;
    p.tma_out = 1;
  }
  // programmatic launch: the block prologue (barriers, TMEM, tensor maps)
  // overlaps the end of the previous kernel; the producers wait for it
  // (griddepcontrol.wait) before their first load.  kInStageKV: blocks wait
  // for flags that other blocks of the grid set, so the grid is launched
  // cooperatively (all blocks resident together; one per multiprocessor)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(P::kThreads);
  cfg.dynamicSmemBytes = P::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if constexpr (kIn == vattn::kInStageKV) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, tql, tkl, tvl, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaErrorCooperativeLaunchTooLarge && coop_refused != nullptr) {
    // not sticky: the caller takes another mode
    (void)cudaGetLastError();
    *coop_refused = true;
    return cuda_fail(e, "cooperative attention kernel launch");
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  return VATTN_OK;
}

template <int NQ, int NKB, bool kOut16 = false>
vattn_status launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              vattn::Params p, unsigned n_tiles, cudaStream_t stream,
                              int device) {
  return launch_attention_maps<NQ, NKB, kOut16, false>(tq, tk, tv, tq, tk, tv, p, n_tiles,
                                                       stream, device);
}

// Query tiles per work tile: two when there is more than one tile of rows
// and the TMEM plan holds two O blocks (d_pad <= 64 with separate P buffers,
// d_pad <= 96 with a shared one), else one.
int query_tiles(int n_patches, int d_pad) {
  return (n_patches > vattn::kBM && d_pad <= 96) ? 2 : 1;
}

// f32 inputs the attention kernel reads directly (its converter warps round
// them to f16 in shared memory, no staging pass): two query tiles, head_dim
// 33..64 and a multiple of 4, 16-byte aligned q, k, v, and n_patches <= 2048;
// and any head_dim <= 64 (a multiple of 4) up to 128 patches, where one
// launch instead of two is what counts.
// Each block rounds the K and V tiles of its own query rows, so a head's
// keys are rounded once per 256 query rows and the shared-memory traffic
// grows with n_patches; measured on GB300 (8 x 16 heads, head_dim 64) the
// single kernel is 1.65x faster than staging + attention at 256 patches,
// 1.23x at 1024, even at 2048 and 0.98x at 2304.  Narrower heads stage
// cheaper (head_dim 32 at 1024 patches: 0.96x), so they keep the two passes.
bool direct_shape(int N, int D) {
  const int d_pad = (D + 15) & ~15;
  if (d_pad > 64 || D % 4 != 0) return false;
  // up to 128 patches (one work tile per head, one key tile): the direct
  // kernel's second query tile reads as zero rows and stores nothing, and
  // the call is one launch instead of a staging pass and the attention kernel
  if (N <= 128) return true;
  return D > 32 && N <= 2048 && query_tiles(N, d_pad) == 2;
}

bool aligned16(const void* q, const void* k, const void* v) {
  return ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
           reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
}

// The attention kernel on f32 inputs (direct_shape and aligned16 hold): one launch;
// p carries the tiling and the work schedule.
vattn_status launch_f32_direct(const float* q, const float* k, const float* v, vattn::Params p,
                               int64_t bh, int N, int D, cudaStream_t stream, int device) {
  CUtensorMap tq, tk, tv;
  vattn_status st;
  if ((st = make_tmap32(&tq, q, bh, N, D)) != VATTN_OK) return st;
  if ((st = make_tmap32(&tk, k, bh, N, D)) != VATTN_OK) return st;
  if ((st = make_tmap32(&tv, v, bh, N, D)) != VATTN_OK) return st;
  return launch_attention_maps<2, 1, false, false, vattn::kInF32>(
      tq, tk, tv, tq, tk, tv, p, static_cast<unsigned>(p.n_tiles), stream, device);
}

// The kernel variant for nkb 64-column blocks of d_pad and nq query tiles.
template <bool kOut16 = false>
vattn_status dispatch_attention(int nkb, int nq, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, vattn::Params p, unsigned g,
                                cudaStream_t stream, int device) {
  if (nkb == 1)
    return nq == 2 ? launch_attention<2, 1, kOut16>(tq, tk, tv, p, g, stream, device)
                   : launch_attention<1, 1, kOut16>(tq, tk, tv, p, g, stream, device);
  return nq == 2 ? launch_attention<2, 2, kOut16>(tq, tk, tv, p, g, stream, device)
                 : launch_attention<1, 2, kOut16>(tq, tk, tv, p, g, stream, device);
}

// Arguments of the NeoX rotation (checked on the host, before any CUDA call).
vattn_status check_rope(int64_t head_dim, int64_t n_patches, int64_t rope_dims, int64_t pos0,
                        float base, const float* factors) {
  if (rope_dims < 0 || rope_dims > head_dim)
    return fail(VATTN_ERR_INVALID_ARG, "rope_dims %lld outside [0, head_dim = %lld]",
                (long long)rope_dims, (long long)head_dim);
  if (!(base > 0.0f) || base > 3.4e38f)
    return fail(VATTN_ERR_INVALID_ARG, "base must be a finite positive number");
  if (pos0 < 0) return fail(VATTN_ERR_INVALID_ARG, "pos0 must be >= 0");
  if (pos0 > (int64_t{1} << 24) - n_patches)
    return fail(VATTN_ERR_UNSUPPORTED,
                "positions up to pos0 + n_patches - 1 must be exact in f32 (< 2^24)");
  if (reinterpret_cast<uintptr_t>(factors) & 3u)
    return fail(VATTN_ERR_MISALIGNED, "factors must be 4-byte aligned");
  return VATTN_OK;
}

bool overlaps(const void* a, const void* b, uint64_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

// [a, a + a_bytes) and [b, b + b_bytes) intersect
bool overlaps2(const void* a, uint64_t a_bytes, const void* b, uint64_t b_bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + b_bytes && y < x + a_bytes;
}

// Size rules of the f32 attention entry points, checked before any CUDA call.
vattn_status check_attention_sizes(int64_t batch, int64_t n_heads, int64_t n_patches,
                                   int64_t head_dim) {
  if (batch < 0 || n_heads < 0 || n_patches < 0 || head_dim < 0)
    return fail(VATTN_ERR_INVALID_ARG, "negative size (batch=%lld n_heads=%lld n_patches=%lld head_dim=%lld)",
                (long long)batch, (long long)n_heads, (long long)n_patches, (long long)head_dim);
  if (head_dim == 0) return fail(VATTN_ERR_INVALID_ARG, "head_dim must be >= 1");
  if (head_dim > VATTN_MAX_HEAD_DIM)
    return fail(VATTN_ERR_UNSUPPORTED, "head_dim %lld > %d", (long long)head_dim, VATTN_MAX_HEAD_DIM);
  return VATTN_OK;
}

// Tensor rules of the f32 attention entry points (sizes already checked):
// *bh receives batch * n_heads; *empty is set, and nothing more checked,
// when there is nothing to compute.
vattn_status check_attention_tensors(const float* q, const float* k, const float* v,
                                     const float* out, int64_t batch, int64_t n_heads,
                                     int64_t n_patches, int64_t head_dim, int64_t* bh,
                                     bool* empty) {
  *empty = false;
  if (batch != 0 && n_heads > INT64_MAX / batch)
    return fail(VATTN_ERR_UNSUPPORTED, "batch * n_heads overflows");
  *bh = batch * n_heads;
  if (*bh == 0 || n_patches == 0) {
    *empty = true;
    return VATTN_OK;
  }
  if (!q || !k || !v || !out) return fail(VATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (n_patches > INT32_MAX || *bh > INT32_MAX)
    return fail(VATTN_ERR_UNSUPPORTED, "n_patches and batch*n_heads must fit in 32 bits");
  if (n_patches > INT64_MAX / head_dim / *bh / 4)
    return fail(VATTN_ERR_UNSUPPORTED, "tensor byte size overflows");
  const uint64_t bytes = static_cast<uint64_t>(*bh) * n_patches * head_dim * 4u;
  const uintptr_t align_or = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                             reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if (align_or & 3u) return fail(VATTN_ERR_MISALIGNED, "tensor pointers must be 4-byte aligned");
  if (overlaps(out, q, bytes) || overlaps(out, k, bytes) || overlaps(out, v, bytes))
    return fail(VATTN_ERR_INVALID_ARG, "out overlaps q, k or v");
  return VATTN_OK;
}

// The attention kernel alone on f16 inputs; out is f32 (kOut16 == false) or
// f16 (kOut16 == true).
template <bool kOut16>
vattn_status forward_f16_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v, void* out,
                              int64_t batch, int64_t n_heads, int64_t n_patches,
                              int64_t head_dim, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks, before any CUDA call
  const vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  if (head_dim % 8 != 0)
    return fail(VATTN_ERR_UNSUPPORTED,
                "f16 inputs need head_dim %% 8 == 0 (16-byte rows), got %lld: use vattn_forward",
                (long long)head_dim);
  if (batch != 0 && n_heads > INT64_MAX / batch)
    return fail(VATTN_ERR_UNSUPPORTED, "batch * n_heads overflows");
  const int64_t bh = batch * n_heads;
  if (bh == 0 || n_patches == 0) return VATTN_OK;  // nothing to compute
  if (!q || !k || !v || !out) return fail(VATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (n_patches > INT32_MAX || bh > INT32_MAX)
    return fail(VATTN_ERR_UNSUPPORTED, "n_patches and batch*n_heads must fit in 32 bits");
  if (n_patches > INT64_MAX / head_dim / bh / 4)
    return fail(VATTN_ERR_UNSUPPORTED, "tensor byte size overflows");
  const uint64_t in_bytes = static_cast<uint64_t>(bh) * n_patches * head_dim * 2u;
  const uint64_t out_bytes = kOut16 ? in_bytes : 2u * in_bytes;
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
        reinterpret_cast<uintptr_t>(v)) & 15u) != 0)
    return fail(VATTN_ERR_MISALIGNED, "f16 q, k, v must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(out) & (kOut16 ? 1u : 3u))
    return fail(VATTN_ERR_MISALIGNED, kOut16 ? "out must be 2-byte aligned" : "out must be 4-byte aligned");
  if (overlaps2(out, out_bytes, q, in_bytes) || overlaps2(out, out_bytes, k, in_bytes) ||
      overlaps2(out, out_bytes, v, in_bytes))
    return fail(VATTN_ERR_INVALID_ARG, "out overlaps q, k or v");

  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int d_pad = (D + 15) & ~15;
  const int nkb = d_pad <= 64 ? 1 : 2;
  const int nq = query_tiles(N, d_pad);
  const int64_t n_qblocks = (N + vattn::kBM * nq - 1) / (vattn::kBM * nq);
  const int64_t grid = bh * n_qblocks;
  if (grid > INT32_MAX) return fail(VATTN_ERR_UNSUPPORTED, "grid too large");

  vattn::Params p{};
  p.out = kOut16 ? nullptr : static_cast<float*>(out);
  p.out16 = kOut16 ? static_cast<uint16_t*>(out) : nullptr;
  p.n_patches = N;
  p.head_dim = D;
  p.d_pad = d_pad;
  p.n_qblocks = static_cast<int>(n_qblocks);
  p.n_tiles = static_cast<int>(grid);
  p.n_ktiles = (N + vattn::kBN - 1) / vattn::kBN;
  p.vec_out = (D % (kOut16 ? 8 : 4) == 0) && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;

  // ---- device side: the tensor maps read the caller's rows of D elements;
  // columns D..d_pad-1 read as zero
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (device < 0 || device >= kMaxDevices) return fail(VATTN_ERR_CUDA, "device index %d out of range", device);
  CUtensorMap tq, tk, tv;
  vattn_status st;
  if ((st = make_tmap16(&tq, reinterpret_cast<const __half*>(q), bh, N, D)) != VATTN_OK) return st;
  if ((st = make_tmap16(&tk, reinterpret_cast<const __half*>(k), bh, N, D)) != VATTN_OK) return st;
  if ((st = make_tmap16(&tv, reinterpret_cast<const __half*>(v), bh, N, D)) != VATTN_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const unsigned g = static_cast<unsigned>(grid);
  return dispatch_attention<kOut16>(nkb, nq, tq, tk, tv, p, g, stream, device);
}

// Blocks of `threads` threads of `kernel` that fit on one multiprocessor,
// looked up once per device (cache: one slot per device).
template <typename Kernel>
vattn_status resident_blocks(Kernel kernel, int threads, int device, std::atomic<int>* cache,
                             int* out) {
  int n = cache[device].load(std::memory_order_acquire);
  if (n <= 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (n <= 0) return fail(VATTN_ERR_CUDA, "kernel does not fit with %d threads per block", threads);
    cache[device].store(n, std::memory_order_release);
  }
  *out = n;
  return VATTN_OK;
}

// The conv1d kernels loop over their items: the grid is what fits on the
// GPU at once (one wave; a grid past that leaves a partial second wave with
// too few loads in flight), fewer blocks for small problems.
template <typename Kernel>
vattn_status launch_streaming(Kernel kernel, std::atomic<int>* cache, long long threads_wanted,
                              const vattn::Conv1dArgs& a, int device, int sms,
                              cudaStream_t stream) {
  int per_sm = 0;
  const vattn_status st = resident_blocks(kernel, 256, device, cache, &per_sm);
  if (st != VATTN_OK) return st;
  const long long blocks = (threads_wanted + 255) / 256;
  const long long cap = static_cast<long long>(per_sm) * sms;
  kernel<<<static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0, stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "conv1d kernel launch");
  return VATTN_OK;
}

template <int DC>
vattn_status launch_conv1d4(const vattn::Conv1dArgs& a, int device, int sms, cudaStream_t stream) {
  static std::atomic<int> cache[2][kMaxDevices];
  const long long items = a.batch * (a.hidden / 4);
  if (a.kernel_size == DC + 1 && (reinterpret_cast<uintptr_t>(a.weight) & 15u) == 0)
    return launch_streaming(vattn::vattn_conv1d_step4_kernel<DC, true>, cache[1], items, a, device,
                            sms, stream);
  return launch_streaming(vattn::vattn_conv1d_step4_kernel<DC, false>, cache[0], items, a, device,
                          sms, stream);
}

// ---------------------------------------------------------------- mode choice
// The single cooperative kernel (k and v staged inside it) needs every block
// of its grid resident at once: the device must support cooperative launches
// and hold one of its 512-thread, ~231 KB blocks per multiprocessor.  Both
// facts are read once per device; vattn_set_single_kernel(0) forbids the mode
// process-wide (the calls then take the two-kernel mode, bit-identical).
struct SingleKernelFacts {
  std::once_flag once;
  int cooperative = 0;    // cudaDevAttrCooperativeLaunch
  int blocks_per_sm = 0;  // resident blocks of the kernel per multiprocessor
  cudaError_t err = cudaSuccess;
};
SingleKernelFacts g_single_facts[kMaxDevices];
std::atomic<int> g_single_kernel_allowed{1};

using SingleKernelPlan = vattn::Plan<2, 1, false, vattn::kInStageKV>;

vattn_status single_kernel_facts(int device, int* cooperative, int* blocks_per_sm) {
  if (device < 0 || device >= kMaxDevices) return fail(VATTN_ERR_CUDA, "device index %d out of range", device);
  SingleKernelFacts& f = g_single_facts[device];
  std::call_once(f.once, [&f, device] {
    f.err = cudaDeviceGetAttribute(&f.cooperative, cudaDevAttrCooperativeLaunch, device);
    if (f.err != cudaSuccess) return;
    auto kernel = vattn::vattn_fwd_kernel<2, 1, false, false, vattn::kInStageKV>;
    // the occupancy query counts dynamic shared memory only up to the
    // kernel's opt-in limit, so raise it first (the launch does the same)
    f.err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SingleKernelPlan::kSmemBytes);
    if (f.err != cudaSuccess) return;
    f.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f.blocks_per_sm, kernel,
                                                          SingleKernelPlan::kThreads,
                                                          SingleKernelPlan::kSmemBytes);
  });
  if (f.err != cudaSuccess) return cuda_fail(f.err, "querying cooperative launch support");
  *cooperative = f.cooperative;
  *blocks_per_sm = f.blocks_per_sm;
  return VATTN_OK;
}

// Up to this many patches a direct shape always takes the direct kernel;
// from 1537 to 2048 patches only while its work tiles fill at most two
// rounds of the grid.  Beyond that the single kernel, which rounds each key
// tile once per head instead of once per query block, measured faster
// (GB300, whole calls: 8 x 16 heads x 2048 x 64 161.6 against 170.1 us,
// 8 x 16 x 1792 x 64 128.5 against 130.9, 4 x 16 x 2048 x 64 97.3 against
// 99.3), and the direct kernel below it (8 x 16 x 1536 x 64 113.6 against
// 114.9, 2 x 16 x 2048 x 64 52.1 against 56.1, 1 x 16 x 2048 x 64 28.6
// against 34.7).
constexpr int kDirectAlwaysMaxN = 1536;

// The kernels a vattn_forward call on a non-empty, valid problem runs, from
// its sizes (n_tiles: its work tiles, batch*n_heads * query blocks), whether
// q, k and v are all 16-byte aligned, and the device facts: n_sms
// multiprocessors (the grid) and the single kernel's facts above
// (single_allowed: the caller and the process-wide switch allow it).
vattn_mode forward_mode_rule(int N, int D, long long n_tiles, int n_sms, bool all_aligned16,
                             bool single_allowed, int cooperative, int blocks_per_sm) {
  const int d_pad = (D + 15) & ~15;
  const int nkb = d_pad <= 64 ? 1 : 2;
  const bool q_f32 = nkb == 1 && query_tiles(N, d_pad) == 2 && D % 4 == 0;
  const bool single = single_allowed && all_aligned16 && q_f32 && cooperative != 0 &&
                      blocks_per_sm >= 1;
  if (all_aligned16 && direct_shape(N, D)) {
    if (single && N > kDirectAlwaysMaxN && n_tiles > 2LL * n_sms) return VATTN_MODE_SINGLE_KERNEL;
    return VATTN_MODE_DIRECT;
  }
  return single ? VATTN_MODE_SINGLE_KERNEL : VATTN_MODE_TWO_KERNELS;
}

// Work tiles of a problem: batch*n_heads * query blocks of nq query tiles.
long long work_tiles(long long bh, int N, int D) {
  const int nq = query_tiles(N, (D + 15) & ~15);
  return bh * ((N + vattn::kBM * nq - 1) / (vattn::kBM * nq));
}

// The mode a call takes on `device` (sizes and pointers already checked).
vattn_status forward_mode_on(int device, const float* q, const float* k, const float* v,
                             int64_t bh, int N, int D, bool single_kernel, vattn_mode* mode) {
  int coop = 0, blocks = 0, sms = 0;
  vattn_status st = sm_count(device, &sms);
  if (st != VATTN_OK) return st;
  const long long n_tiles = work_tiles(bh, N, D);
  const bool allowed = single_kernel && g_single_kernel_allowed.load(std::memory_order_relaxed) != 0;
  const bool al = aligned16(q, k, v);
  // the facts are read only when the rule could take the single kernel
  if (allowed &&
      forward_mode_rule(N, D, n_tiles, sms, al, true, 1, 1) == VATTN_MODE_SINGLE_KERNEL) {
    st = single_kernel_facts(device, &coop, &blocks);
    if (st != VATTN_OK) return st;
  }
  *mode = forward_mode_rule(N, D, n_tiles, sms, al, allowed, coop, blocks);
  return VATTN_OK;
}

// Everything a vattn_forward call decides before it launches: the mode, the
// tiling, the work schedule and the workspace it needs, laid out as
//   sync words | partial slots | f16 q | f16 k | f16 v
// Sync words: two per (cut slot, query tile, softmax warp) -- arrival
// count, ready flag --
// then, in the single kernel's mode, one ready flag per (head, key tile);
// one memset per call clears them.  Partial slots: one per block boundary
// of a cut schedule.  The f16 copies: none in the direct mode.
struct ForwardPlan {
  vattn_mode mode = VATTN_MODE_TWO_KERNELS;
  int N = 0, D = 0, d_pad = 0, nkb = 1, nq = 1, T = 0, grid = 0;
  int64_t bh = 0, n_qblocks = 0, n_tiles = 0;
  Schedule sched;
  size_t cut_words = 0, flag_words = 0;
  size_t sync_bytes = 0;  // 256-byte rounded
  size_t part_bytes = 0;  // 256-byte rounded
  size_t region = 0;      // one f16 copy, 256-byte rounded (0: none)
  size_t total() const { return sync_bytes + part_bytes + 3 * region; }
};

size_t round256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

// Blocks of 256 threads per tensor for the staging kernels (one row of
// blocks per tensor, n_tensors rows): one thread per 8-column chunk, at most
// 16 blocks per multiprocessor of 152 in all rows together (the threads then
// walk several chunks each).
unsigned stage_blocks(long long chunks_per_tensor, unsigned n_tensors) {
  const long long cap = 152LL * 16 / n_tensors;
  const long long blocks = (chunks_per_tensor + 255) / 256;
  return static_cast<unsigned>(blocks < cap ? blocks : cap);
}

// single_kernel: the caller allows the single cooperative kernel (the
// host-buffer entry point does not); max_sync_part_bytes: room for the sync
// words and partial slots together (a cut schedule is taken only if they
// fit; 0: never).  Arguments are valid and the problem is not empty
// (checked by the entry points).
vattn_status plan_forward(int device, const float* q, const float* k, const float* v, int64_t bh,
                          int N, int D, bool single_kernel, size_t max_sync_part_bytes,
                          ForwardPlan* out) {
  ForwardPlan pl;
  vattn_status st = forward_mode_on(device, q, k, v, bh, N, D, single_kernel, &pl.mode);
  if (st != VATTN_OK) return st;
  pl.N = N;
  pl.D = D;
  pl.bh = bh;
  pl.d_pad = (D + 15) & ~15;
  pl.nkb = pl.d_pad <= 64 ? 1 : 2;
  pl.nq = query_tiles(N, pl.d_pad);
  pl.n_qblocks = (N + vattn::kBM * pl.nq - 1) / (vattn::kBM * pl.nq);
  pl.n_tiles = bh * pl.n_qblocks;
  if (pl.n_tiles > INT32_MAX) return fail(VATTN_ERR_UNSUPPORTED, "grid too large");
  pl.T = (N + vattn::kBN - 1) / vattn::kBN;
  int sms = 0;
  if ((st = sm_count(device, &sms)) != VATTN_OK) return st;
  pl.grid = static_cast<int>(pl.n_tiles < sms ? pl.n_tiles : sms);
  if (pl.mode == VATTN_MODE_SINGLE_KERNEL) pl.flag_words = static_cast<size_t>(bh) * pl.T;
  const size_t slot_bytes = part_slot_floats(pl.nq, pl.d_pad) * sizeof(float);
  const size_t cut_words = static_cast<size_t>(pl.grid - 1) * pl.nq * 4 * 2;
  const size_t cut_need = round256((cut_words + pl.flag_words) * sizeof(uint32_t)) +
                          round256(static_cast<size_t>(pl.grid - 1) * slot_bytes);
  pl.sched = make_schedule(pl.n_tiles, pl.T, pl.grid,
                           cut_need <= max_sync_part_bytes
                               ? g_cut_allowed.load(std::memory_order_relaxed) : 0);
  if (pl.sched.cut) {
    pl.cut_words = cut_words;
    pl.part_bytes = round256(static_cast<size_t>(pl.grid - 1) * slot_bytes);
  }
  pl.sync_bytes = round256((pl.cut_words + pl.flag_words) * sizeof(uint32_t));
  if (pl.mode != VATTN_MODE_DIRECT)
    pl.region = round256(static_cast<size_t>(bh) * N * pl.d_pad * 2);
  *out = pl;
  return VATTN_OK;
}

// The kernels of a planned vattn_forward call: sync (plan.sync_bytes) and
// part (plan.part_bytes) and staging (3 regions of plan.region) are the
// caller's workspace.  One memset clears the sync words; then the direct
// f32 kernel, or the single cooperative kernel, or the staging kernel and
// the attention kernel.  With two query tiles of head_dim <= 64 the
// attention kernel reads q in f32 and rounds it itself (q is read once per
// work tile, so that costs it little) and the staging kernel rounds k and v
// alone.  A cooperative grid that the device refuses at launch (for example
// under an MPS limit on multiprocessors) gets the two kernels instead.
vattn_status run_forward(const ForwardPlan& pl, const float* q, const float* k, const float* v,
                         float* out, uint32_t* sync, float* part, void* staging,
                         cudaStream_t stream, int device) {
  const int N = pl.N, D = pl.D, d_pad = pl.d_pad, nkb = pl.nkb, nq = pl.nq;
  const int64_t bh = pl.bh;
  if (pl.sync_bytes > 0) {
    const cudaError_t e = cudaMemsetAsync(sync, 0, pl.sync_bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace flags");
  }
  vattn::Params p{};
  p.out = out;
  p.n_patches = N;
  p.head_dim = D;
  p.d_pad = d_pad;
  p.n_qblocks = static_cast<int>(pl.n_qblocks);
  p.n_tiles = static_cast<int>(pl.n_tiles);
  p.n_ktiles = pl.T;
  p.vec_out = (D % 4 == 0) && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  p.rounds = pl.sched.rounds;
  p.extra = pl.sched.extra;
  p.tail_units = pl.sched.tail_units;
  p.part = pl.sched.cut ? part : nullptr;
  p.part_sync = pl.sched.cut ? sync : nullptr;
  if (pl.mode == VATTN_MODE_DIRECT) return launch_f32_direct(q, k, v, p, bh, N, D, stream, device);
  const int64_t grid = pl.n_tiles;
  const bool q_f32 = nkb == 1 && nq == 2 && D % 4 == 0 && (reinterpret_cast<uintptr_t>(q) & 15u) == 0;
  __half* q16 = static_cast<__half*>(staging);
  __half* k16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(staging) + pl.region);
  __half* v16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(staging) + 2 * pl.region);
  CUtensorMap tq, tk, tv;
  vattn_status st;
  if ((st = q_f32 ? make_tmap32(&tq, q, bh, N, D) : make_tmap16(&tq, q16, bh, N, d_pad)) != VATTN_OK)
    return st;
  if ((st = make_tmap16(&tk, k16, bh, N, d_pad)) != VATTN_OK) return st;
  if ((st = make_tmap16(&tv, v16, bh, N, d_pad)) != VATTN_OK) return st;
  if (pl.mode == VATTN_MODE_SINGLE_KERNEL) {
    // one kernel: it writes the f16 copies of k and v itself, each key tile
    // once, and the blocks that read a tile wait for its ready flag (after
    // the cut-tile words in the sync block)
    p.k16 = reinterpret_cast<uint16_t*>(k16);
    p.v16 = reinterpret_cast<uint16_t*>(v16);
    p.kv_ready = sync + pl.cut_words;
    CUtensorMap tk32, tv32;  // the f32 tiles the kernel stages from
    vattn_status sm;
    if ((sm = make_tmap32(&tk32, k, bh, N, D)) != VATTN_OK) return sm;
    if ((sm = make_tmap32(&tv32, v, bh, N, D)) != VATTN_OK) return sm;
    bool refused = false;
    sm = launch_attention_maps<2, 1, false, false, vattn::kInStageKV>(
        tq, tk, tv, tq, tk32, tv32, p, static_cast<unsigned>(grid), stream, device, &refused);
    if (!refused) return sm;
    g_last_error[0] = '\0';
    p.k16 = p.v16 = nullptr;
    p.kv_ready = nullptr;
  }
  const int64_t rows = bh * N;
  const uintptr_t src_or = (q_f32 ? 0u : reinterpret_cast<uintptr_t>(q)) |
                           reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v);
  const int vec = (D % 8 == 0) && (src_or & 15u) == 0;
  const unsigned n_jobs = q_f32 ? 2u : 3u;
  const dim3 stage_grid(stage_blocks(rows * (d_pad / 8), n_jobs), n_jobs);
  if (q_f32)
    vattn::vattn_stage_kernel<<<stage_grid, 256, 0, stream>>>(
        vattn::StageJob{k, k16}, vattn::StageJob{v, v16}, vattn::StageJob{nullptr, nullptr}, rows,
        D, d_pad, vec);
  else
    vattn::vattn_stage_kernel<<<stage_grid, 256, 0, stream>>>(
        vattn::StageJob{q, q16}, vattn::StageJob{k, k16}, vattn::StageJob{v, v16}, rows, D, d_pad,
        vec);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "staging kernel launch");
  const unsigned g = static_cast<unsigned>(grid);
  if (q_f32)
    return launch_attention_maps<2, 1, false, false, vattn::kInF32Q>(tq, tk, tv, tq, tk, tv, p, g,
                                                                      stream, device);
  return dispatch_attention(nkb, nq, tq, tk, tv, p, g, stream, device);
}

// Most chunks of heads a host-buffer call is cut into (measured on the
// 8x16x2304x64 workload: 4 chunks 1.37 ms, 8 chunks 1.34 ms, 16 chunks
// 1.43 ms per call).
constexpr int64_t kHostChunks = 8;

// Three internal streams per device for the host-buffer entry point: host
// to device copies, kernels, device to host copies.
struct HostStreams {
  std::once_flag once;
  cudaStream_t s[3] = {nullptr, nullptr, nullptr};
  cudaError_t err = cudaSuccess;
};
HostStreams g_host_streams[kMaxDevices];

vattn_status host_streams(int device, cudaStream_t** out) {
  if (device < 0 || device >= kMaxDevices) return fail(VATTN_ERR_CUDA, "device index %d out of range", device);
  HostStreams& hs = g_host_streams[device];
  std::call_once(hs.once, [&hs] {
    for (int i = 0; i < 3 && hs.err == cudaSuccess; ++i)
      hs.err = cudaStreamCreateWithFlags(&hs.s[i], cudaStreamNonBlocking);
  });
  if (hs.err != cudaSuccess) return cuda_fail(hs.err, "creating the copy and compute streams");
  *out = hs.s;
  return VATTN_OK;
}

// Wait site reported by the self-test of the timeout path.
constexpr uint32_t kSiteSelfTest = 15;

// One thread waits, with the kernels' bounded wait, for phase 0 of an
// mbarrier that nothing arrives on: after the wait limit it records a
// timeout in the status word, exactly as a stalled attention kernel would,
// and returns.
__global__ void vattn_selftest_wait_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    vattn::ptx::mbar_init(vattn::ptx::smem_addr(&bar), 1);
    abort_flag = 0;
    vattn::ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const vattn::Waiter w{&abort_flag};
    w.wait(vattn::ptx::smem_addr(&bar), 0u, kSiteSelfTest);
  }
}

}  // namespace

extern "C" {

vattn_status vattn_forward(const float* q, const float* k, const float* v, float* out,
                           int64_t batch, int64_t n_heads, int64_t n_patches, int64_t head_dim,
                           void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks, before any CUDA call
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  int64_t bh = 0;
  bool empty = false;
  chk = check_attention_tensors(q, k, v, out, batch, n_heads, n_patches, head_dim, &bh, &empty);
  if (chk != VATTN_OK) return chk;
  if (empty) return VATTN_OK;  // nothing to compute
  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int d_pad = (D + 15) & ~15;

  // ---- device side
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  (void)d_pad;
  ForwardPlan pl;
  vattn_status st = plan_forward(device, q, k, v, bh, N, D, true, SIZE_MAX, &pl);
  if (st != VATTN_OK) return st;
  if (pl.total() == 0) return run_forward(pl, q, k, v, out, nullptr, nullptr, nullptr, stream, device);

  // sync words, partial slots and f16 copies: stream-ordered workspace
  cudaMemPool_t pool = nullptr;
  if ((st = pool_for(device, &pool)) != VATTN_OK) return st;
  void* ws = nullptr;
  e = cudaMallocFromPoolAsync(&ws, pl.total(), pool, stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  uint8_t* const wb = static_cast<uint8_t*>(ws);
  st = run_forward(pl, q, k, v, out, reinterpret_cast<uint32_t*>(wb),
                   reinterpret_cast<float*>(wb + pl.sync_bytes), wb + pl.sync_bytes + pl.part_bytes,
                   stream, device);
  // back to the pool once the launches above have run (stream order)
  e = cudaFreeAsync(ws, stream);
  if (st == VATTN_OK && e != cudaSuccess) st = cuda_fail(e, "workspace release");
  return st;
}

vattn_status vattn_forward_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               float* out, int64_t batch, int64_t n_heads, int64_t n_patches,
                               int64_t head_dim, void* stream_ptr) {
  return forward_f16_impl<false>(q, k, v, out, batch, n_heads, n_patches, head_dim, stream_ptr);
}

vattn_status vattn_forward_f16io(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* out, int64_t batch, int64_t n_heads,
                                 int64_t n_patches, int64_t head_dim, void* stream_ptr) {
  return forward_f16_impl<true>(q, k, v, out, batch, n_heads, n_patches, head_dim, stream_ptr);
}

vattn_status vattn_forward_f32q(const float* q, const uint16_t* k, const uint16_t* v, float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks, before any CUDA call
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  if (head_dim % 8 != 0 || head_dim > 64)
    return fail(VATTN_ERR_UNSUPPORTED,
                "f32 q with f16 k, v needs head_dim %% 8 == 0 and <= 64, got %lld: use "
                "vattn_forward_f16 with q rounded to f16",
                (long long)head_dim);
  if (batch != 0 && n_heads > INT64_MAX / batch)
    return fail(VATTN_ERR_UNSUPPORTED, "batch * n_heads overflows");
  const int64_t bh = batch * n_heads;
  if (bh == 0 || n_patches == 0) return VATTN_OK;  // nothing to compute
  if (n_patches <= vattn::kBM)
    return fail(VATTN_ERR_UNSUPPORTED,
                "f32 q with f16 k, v needs n_patches > %d, got %lld: use vattn_forward_f16 with q "
                "rounded to f16",
                vattn::kBM, (long long)n_patches);
  if (!q || !k || !v || !out) return fail(VATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (n_patches > INT32_MAX || bh > INT32_MAX)
    return fail(VATTN_ERR_UNSUPPORTED, "n_patches and batch*n_heads must fit in 32 bits");
  if (n_patches > INT64_MAX / head_dim / bh / 4)
    return fail(VATTN_ERR_UNSUPPORTED, "tensor byte size overflows");
  const uint64_t f32_bytes = static_cast<uint64_t>(bh) * n_patches * head_dim * 4u;
  const uint64_t f16_bytes = f32_bytes / 2u;
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
        reinterpret_cast<uintptr_t>(v)) & 15u) != 0)
    return fail(VATTN_ERR_MISALIGNED, "q, k, v must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(out) & 3u)
    return fail(VATTN_ERR_MISALIGNED, "out must be 4-byte aligned");
  if (overlaps(out, q, f32_bytes) || overlaps2(out, f32_bytes, k, f16_bytes) ||
      overlaps2(out, f32_bytes, v, f16_bytes))
    return fail(VATTN_ERR_INVALID_ARG, "out overlaps q, k or v");

  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int64_t n_qblocks = (N + 2 * vattn::kBM - 1) / (2 * vattn::kBM);
  const int64_t grid = bh * n_qblocks;
  if (grid > INT32_MAX) return fail(VATTN_ERR_UNSUPPORTED, "grid too large");
  vattn::Params p{};
  p.out = out;
  p.n_patches = N;
  p.head_dim = D;
  p.d_pad = (D + 15) & ~15;
  p.n_qblocks = static_cast<int>(n_qblocks);
  p.n_tiles = static_cast<int>(grid);
  p.n_ktiles = (N + vattn::kBN - 1) / vattn::kBN;
  p.vec_out = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;

  // ---- device side
  int device = 0;
  const cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  CUtensorMap tq, tk, tv;
  vattn_status st;
  if ((st = make_tmap32(&tq, q, bh, N, D)) != VATTN_OK) return st;
  if ((st = make_tmap16(&tk, reinterpret_cast<const __half*>(k), bh, N, D)) != VATTN_OK) return st;
  if ((st = make_tmap16(&tv, reinterpret_cast<const __half*>(v), bh, N, D)) != VATTN_OK) return st;
  return launch_attention_maps<2, 1, false, false, vattn::kInF32Q>(
      tq, tk, tv, tq, tk, tv, p, static_cast<unsigned>(grid), static_cast<cudaStream_t>(stream_ptr),
      device);
}

vattn_status vattn_rope_neox(float* x, int64_t batch, int64_t n_heads, int64_t n_patches,
                             int64_t head_dim, int64_t rope_dims, int64_t pos0, float base,
                             const float* factors, int inverse, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks, before any CUDA call
  if (batch < 0 || n_heads < 0 || n_patches < 0 || head_dim < 0)
    return fail(VATTN_ERR_INVALID_ARG, "negative size");
  if (head_dim == 0) return fail(VATTN_ERR_INVALID_ARG, "head_dim must be >= 1");
  if (inverse != 0 && inverse != 1) return fail(VATTN_ERR_INVALID_ARG, "inverse must be 0 or 1");
  vattn_status st = check_rope(head_dim, n_patches, rope_dims, pos0, base, factors);
  if (st != VATTN_OK) return st;
  if (batch != 0 && n_heads > INT64_MAX / batch)
    return fail(VATTN_ERR_UNSUPPORTED, "batch * n_heads overflows");
  const int64_t bh = batch * n_heads;
  const int half = static_cast<int>(rope_dims / 2);
  if (bh == 0 || n_patches == 0 || half == 0) return VATTN_OK;  // nothing turns
  if (!x) return fail(VATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (n_patches > INT32_MAX || bh > INT64_MAX / n_patches || bh * n_patches > INT64_MAX / head_dim)
    return fail(VATTN_ERR_UNSUPPORTED, "tensor size overflows");
  if (reinterpret_cast<uintptr_t>(x) & 3u)
    return fail(VATTN_ERR_MISALIGNED, "x must be 4-byte aligned");

  // ---- device side: angle table (stream-ordered workspace), then the turn
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaMemPool_t pool = nullptr;
  if ((st = pool_for(device, &pool)) != VATTN_OK) return st;
  void* tab = nullptr;
  e = cudaMallocFromPoolAsync(&tab, static_cast<size_t>(n_patches) * half * sizeof(float2), pool,
                              stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  const int N = static_cast<int>(n_patches);
  auto grid_for = [](long long items) {
    const long long blocks = (items + 255) / 256;
    return static_cast<unsigned>(blocks < 152LL * 16 ? blocks : 152LL * 16);
  };
  vattn::vattn_rope_table_kernel<<<grid_for(static_cast<long long>(N) * half), 256, 0, stream>>>(
      static_cast<float2*>(tab), N, half, static_cast<int>(rope_dims), pos0, base, factors);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    st = cuda_fail(e, "RoPE table kernel launch");
  } else {
    const long long rows = bh * n_patches;
    const bool by4 = (half % 4 == 0) && (head_dim % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    if (by4)
      vattn::vattn_rope_apply4_kernel<<<grid_for(rows * (half / 4)), 256, 0, stream>>>(
          x, rows, N, static_cast<int>(head_dim), half, static_cast<const float2*>(tab), inverse);
    else
      vattn::vattn_rope_apply_kernel<<<grid_for(rows * half), 256, 0, stream>>>(
          x, rows, N, static_cast<int>(head_dim), half, static_cast<const float2*>(tab), inverse);
    e = cudaGetLastError();
    if (e != cudaSuccess) st = cuda_fail(e, "RoPE kernel launch");
  }
  e = cudaFreeAsync(tab, stream);
  if (st == VATTN_OK && e != cudaSuccess) st = cuda_fail(e, "workspace release");
  return st;
}

vattn_status vattn_forward_rope(const float* q, const float* k, const float* v, float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, int64_t rope_dims, int64_t pos0, float base,
                                const float* factors, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks (those of vattn_forward and of the rotation)
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  chk = check_rope(head_dim, n_patches, rope_dims, pos0, base, factors);
  if (chk != VATTN_OK) return chk;
  int64_t bh = 0;
  bool empty = false;
  chk = check_attention_tensors(q, k, v, out, batch, n_heads, n_patches, head_dim, &bh, &empty);
  if (chk != VATTN_OK) return chk;
  if (empty) return VATTN_OK;  // nothing to compute

  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int d_pad = (D + 15) & ~15;
  const int half = static_cast<int>(rope_dims / 2);
  const int nkb = d_pad <= 64 ? 1 : 2;
  const int nq = query_tiles(N, d_pad);
  const int64_t n_qblocks = (N + vattn::kBM * nq - 1) / (vattn::kBM * nq);
  const int64_t grid = bh * n_qblocks;
  if (grid > INT32_MAX) return fail(VATTN_ERR_UNSUPPORTED, "grid too large");
  vattn::Params p{};
  p.out = out;
  p.n_patches = N;
  p.head_dim = D;
  p.d_pad = d_pad;
  p.n_qblocks = static_cast<int>(n_qblocks);
  p.n_tiles = static_cast<int>(grid);
  p.n_ktiles = (N + vattn::kBN - 1) / vattn::kBN;
  p.vec_out = (D % 4 == 0) && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;

  // ---- device side: workspace = f16 copies of q, k, v + the angle table
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t rows = bh * N;
  const size_t region = (static_cast<size_t>(rows) * d_pad * 2 + 255) & ~static_cast<size_t>(255);
  const size_t tab_bytes = static_cast<size_t>(N) * (half > 0 ? half : 1) * sizeof(float2);
  cudaMemPool_t pool = nullptr;
  vattn_status st = pool_for(device, &pool);
  if (st != VATTN_OK) return st;
  void* ws = nullptr;
  e = cudaMallocFromPoolAsync(&ws, 3 * region + tab_bytes, pool, stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  __half* q16 = static_cast<__half*>(ws);
  __half* k16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) + region);
  __half* v16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) + 2 * region);
  float2* tab = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + 3 * region);

  CUtensorMap tq, tk, tv;
  if ((st = make_tmap16(&tq, q16, bh, N, d_pad)) == VATTN_OK &&
      (st = make_tmap16(&tk, k16, bh, N, d_pad)) == VATTN_OK &&
      (st = make_tmap16(&tv, v16, bh, N, d_pad)) == VATTN_OK) {
    auto grid_for = [](long long items) {
      const long long blocks = (items + 255) / 256;
      return static_cast<unsigned>(blocks < 152LL * 16 ? blocks : 152LL * 16);
    };
    if (half > 0) {
      vattn::vattn_rope_table_kernel<<<grid_for(static_cast<long long>(N) * half), 256, 0, stream>>>(
          tab, N, half, static_cast<int>(rope_dims), pos0, base, factors);
      e = cudaGetLastError();
      if (e != cudaSuccess) st = cuda_fail(e, "RoPE table kernel launch");
    }
    const int vec = (D % 8 == 0) &&
                    ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                      reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
    if (st == VATTN_OK) {
      vattn::vattn_stage_rope_kernel<<<grid_for(3LL * rows * (d_pad / 8)), 256, 0, stream>>>(
          vattn::StageJob{q, q16}, vattn::StageJob{k, k16}, vattn::StageJob{v, v16}, rows, N, D,
          d_pad, half, tab, vec);
      e = cudaGetLastError();
      if (e != cudaSuccess) st = cuda_fail(e, "staging kernel launch");
    }
    if (st == VATTN_OK) {
      const unsigned g = static_cast<unsigned>(grid);
      st = dispatch_attention(nkb, nq, tq, tk, tv, p, g, stream, device);
    }
  }
  e = cudaFreeAsync(ws, stream);
  if (st == VATTN_OK && e != cudaSuccess) st = cuda_fail(e, "workspace release");
  return st;
}

vattn_status vattn_forward_accurate(const float* q, const float* k, const float* v, float* out,
                                    int64_t batch, int64_t n_heads, int64_t n_patches,
                                    int64_t head_dim, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks: those of vattn_forward
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  int64_t bh = 0;
  bool empty = false;
  chk = check_attention_tensors(q, k, v, out, batch, n_heads, n_patches, head_dim, &bh, &empty);
  if (chk != VATTN_OK) return chk;
  if (empty) return VATTN_OK;  // nothing to compute

  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int d_pad = (D + 15) & ~15;
  const int nkb = d_pad <= 64 ? 1 : 2;
  const int64_t n_qblocks = (N + vattn::kBM - 1) / vattn::kBM;  // one query tile per work tile
  const int64_t grid = bh * n_qblocks;
  if (grid > INT32_MAX) return fail(VATTN_ERR_UNSUPPORTED, "grid too large");
  vattn::Params p{};
  p.out = out;
  p.n_patches = N;
  p.head_dim = D;
  p.d_pad = d_pad;
  p.n_qblocks = static_cast<int>(n_qblocks);
  p.n_tiles = static_cast<int>(grid);
  p.n_ktiles = (N + vattn::kBN - 1) / vattn::kBN;
  p.vec_out = (D % 4 == 0) && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;

  // ---- device side: workspace = f16 hi and lo copies of q, k, v
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t rows = bh * N;
  const size_t region = (static_cast<size_t>(rows) * d_pad * 2 + 255) & ~static_cast<size_t>(255);
  cudaMemPool_t pool = nullptr;
  vattn_status st = pool_for(device, &pool);
  if (st != VATTN_OK) return st;
  void* ws = nullptr;
  e = cudaMallocFromPoolAsync(&ws, 6 * region, pool, stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  __half* part[6];
  for (int i = 0; i < 6; ++i)
    part[i] = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) + i * region);
  CUtensorMap tm[6];
  for (int i = 0; i < 6 && st == VATTN_OK; ++i) st = make_tmap16(&tm[i], part[i], bh, N, d_pad);
  if (st == VATTN_OK) {
    const int vec = (D % 8 == 0) &&
                    ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                      reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
    const dim3 stage_grid(stage_blocks(rows * (d_pad / 8), 3), 3);
    vattn::vattn_stage_split_kernel<<<stage_grid, 256, 0, stream>>>(
        vattn::SplitJob{q, part[0], part[3]}, vattn::SplitJob{k, part[1], part[4]},
        vattn::SplitJob{v, part[2], part[5]}, rows, D, d_pad, vec);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      st = cuda_fail(e, "staging kernel launch");
    } else {
      const unsigned g = static_cast<unsigned>(grid);
      if (nkb == 1)
        st = launch_attention_maps<1, 1, false, true>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], p,
                                                      g, stream, device);
      else
        st = launch_attention_maps<1, 2, false, true>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], p,
                                                      g, stream, device);
    }
  }
  e = cudaFreeAsync(ws, stream);
  if (st == VATTN_OK && e != cudaSuccess) st = cuda_fail(e, "workspace release");
  return st;
}

vattn_status vattn_conv1d_step(const float* input, float* buffer, const float* weight,
                               float* output, int64_t batch, int64_t hidden_size,
                               int64_t kernel_size, int64_t d_conv, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks, before any CUDA call
  if (batch < 0 || hidden_size < 0 || kernel_size < 0 || d_conv < 0)
    return fail(VATTN_ERR_INVALID_ARG, "negative size (batch=%lld hidden_size=%lld kernel_size=%lld d_conv=%lld)",
                (long long)batch, (long long)hidden_size, (long long)kernel_size, (long long)d_conv);
  if (kernel_size < d_conv + 1)
    return fail(VATTN_ERR_INVALID_ARG, "kernel_size %lld < d_conv + 1 = %lld (tap d_conv weighs the input)",
                (long long)kernel_size, (long long)d_conv + 1);
  if (hidden_size > INT32_MAX || kernel_size > INT32_MAX || d_conv > INT32_MAX)
    return fail(VATTN_ERR_UNSUPPORTED, "hidden_size, kernel_size and d_conv must fit in 32 bits");
  if (batch == 0 || hidden_size == 0) return VATTN_OK;  // nothing to compute
  if (!input || !weight || !output || (d_conv > 0 && !buffer))
    return fail(VATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (batch > INT64_MAX / 4 / hidden_size / (d_conv + 1) || hidden_size > INT64_MAX / 4 / kernel_size)
    return fail(VATTN_ERR_UNSUPPORTED, "tensor byte size overflows");
  const uint64_t row_bytes = static_cast<uint64_t>(batch) * hidden_size * 4u;
  const uint64_t buf_bytes = row_bytes * static_cast<uint64_t>(d_conv);
  const uint64_t w_bytes = static_cast<uint64_t>(hidden_size) * kernel_size * 4u;
  const uintptr_t align_or = reinterpret_cast<uintptr_t>(input) | reinterpret_cast<uintptr_t>(buffer) |
                             reinterpret_cast<uintptr_t>(weight) | reinterpret_cast<uintptr_t>(output);
  if (align_or & 3u) return fail(VATTN_ERR_MISALIGNED, "tensor pointers must be 4-byte aligned");
  if (overlaps2(output, row_bytes, input, row_bytes) || overlaps2(output, row_bytes, weight, w_bytes) ||
      (d_conv > 0 && overlaps2(output, row_bytes, buffer, buf_bytes)))
    return fail(VATTN_ERR_INVALID_ARG, "output overlaps input, buffer or weight");
  if (d_conv > 0 && (overlaps2(buffer, buf_bytes, input, row_bytes) ||
                     overlaps2(buffer, buf_bytes, weight, w_bytes)))
    return fail(VATTN_ERR_INVALID_ARG, "buffer overlaps input or weight");

  // ---- device side: one streaming kernel
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int sms = 0;
  const vattn_status st = sm_count(device, &sms);
  if (st != VATTN_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  vattn::Conv1dArgs a{input, buffer, weight, output, static_cast<long long>(batch),
                      static_cast<int>(hidden_size), static_cast<int>(kernel_size),
                      static_cast<int>(d_conv)};
  const bool by4 = (hidden_size % 4 == 0) && d_conv <= 8 &&
                   ((reinterpret_cast<uintptr_t>(input) | reinterpret_cast<uintptr_t>(buffer) |
                     reinterpret_cast<uintptr_t>(output)) & 15u) == 0;
  if (!by4) {
    static std::atomic<int> cache[kMaxDevices];
    return launch_streaming(vattn::vattn_conv1d_step_kernel, cache, batch * hidden_size, a, device,
                            sms, stream);
  }
  switch (d_conv) {
    case 0: return launch_conv1d4<0>(a, device, sms, stream);
    case 1: return launch_conv1d4<1>(a, device, sms, stream);
    case 2: return launch_conv1d4<2>(a, device, sms, stream);
    case 3: return launch_conv1d4<3>(a, device, sms, stream);
    case 4: return launch_conv1d4<4>(a, device, sms, stream);
    case 5: return launch_conv1d4<5>(a, device, sms, stream);
    case 6: return launch_conv1d4<6>(a, device, sms, stream);
    case 7: return launch_conv1d4<7>(a, device, sms, stream);
    default: return launch_conv1d4<8>(a, device, sms, stream);
  }
}

vattn_status vattn_forward_host(const float* q, const float* k, const float* v, float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks: those of vattn_forward
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  int64_t bh = 0;
  bool empty = false;
  chk = check_attention_tensors(q, k, v, out, batch, n_heads, n_patches, head_dim, &bh, &empty);
  if (chk != VATTN_OK) return chk;
  if (empty) return VATTN_OK;  // nothing to compute

  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int d_pad = (D + 15) & ~15;
  // chunks of whole heads, so that copies in, kernels and copies out of
  // consecutive chunks overlap
  const int64_t hc = (bh + kHostChunks - 1) / kHostChunks;  // heads per chunk (the last may have fewer)
  const int64_t n_chunks = (bh + hc - 1) / hc;               // 1..kHostChunks, none empty
  const uint64_t head_bytes = static_cast<uint64_t>(N) * D * 4u;
  const auto round256 = [](uint64_t x) { return (x + 255u) & ~static_cast<uint64_t>(255u); };
  const uint64_t in_slot = 3 * round256(hc * head_bytes);  // f32 q, k, v of one chunk
  const uint64_t out_slot = round256(hc * head_bytes);
  const uint64_t region = round256(static_cast<uint64_t>(hc) * N * d_pad * 2u);  // f16 staging
  const uint64_t ws_bytes = 2 * in_slot + 2 * out_slot + 3 * region;

  // ---- device side
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaStream_t* hs = nullptr;
  vattn_status st = host_streams(device, &hs);
  if (st != VATTN_OK) return st;
  cudaMemPool_t pool = nullptr;
  if ((st = pool_for(device, &pool)) != VATTN_OK) return st;
  void* ws = nullptr;
  e = cudaMallocFromPoolAsync(&ws, ws_bytes, pool, stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  uint8_t* const base = static_cast<uint8_t*>(ws);
  auto in_ptr = [&](int64_t c, int which) {
    return reinterpret_cast<float*>(base + (c & 1) * in_slot + which * round256(hc * head_bytes));
  };
  auto out_ptr = [&](int64_t c) { return reinterpret_cast<float*>(base + 2 * in_slot + (c & 1) * out_slot); };
  void* const ws16 = base + 2 * in_slot + 2 * out_slot;

  // events: start, and per chunk copies in / kernels / copy out done
  cudaEvent_t ev[1 + 3 * kHostChunks] = {};
  int n_ev = 0;
  for (; n_ev < 1 + 3 * n_chunks && st == VATTN_OK; ++n_ev) {
    e = cudaEventCreateWithFlags(&ev[n_ev], cudaEventDisableTiming);
    if (e != cudaSuccess) st = cuda_fail(e, "cudaEventCreate");
  }
  cudaEvent_t* ev_in = ev + 1;
  cudaEvent_t* ev_comp = ev + 1 + n_chunks;
  cudaEvent_t* ev_out = ev + 1 + 2 * n_chunks;
  const cudaStream_t s_in = hs[0], s_comp = hs[1], s_out = hs[2];
  auto ck = [&](cudaError_t err, const char* what) {
    if (st == VATTN_OK && err != cudaSuccess) st = cuda_fail(err, what);
    return st == VATTN_OK;
  };
  bool joined = false;
  if (st == VATTN_OK && ck(cudaEventRecord(ev[0], stream), "cudaEventRecord") &&
      ck(cudaStreamWaitEvent(s_in, ev[0], 0), "cudaStreamWaitEvent") &&
      ck(cudaStreamWaitEvent(s_comp, ev[0], 0), "cudaStreamWaitEvent") &&
      ck(cudaStreamWaitEvent(s_out, ev[0], 0), "cudaStreamWaitEvent")) {
    for (int64_t c = 0; c < n_chunks && st == VATTN_OK; ++c) {
      const int64_t h0 = c * hc;
      const int64_t hn = (h0 + hc <= bh) ? hc : bh - h0;
      const size_t nb = static_cast<size_t>(hn * head_bytes);
      const size_t off = static_cast<size_t>(h0) * N * D;  // elements
      // copies in; the slot is free once the kernels of chunk c - 2 ran
      if (c >= 2 && !ck(cudaStreamWaitEvent(s_in, ev_comp[c - 2], 0), "cudaStreamWaitEvent")) break;
      if (!ck(cudaMemcpyAsync(in_ptr(c, 0), q + off, nb, cudaMemcpyHostToDevice, s_in), "copy of q") ||
          !ck(cudaMemcpyAsync(in_ptr(c, 1), k + off, nb, cudaMemcpyHostToDevice, s_in), "copy of k") ||
          !ck(cudaMemcpyAsync(in_ptr(c, 2), v + off, nb, cudaMemcpyHostToDevice, s_in), "copy of v") ||
          !ck(cudaEventRecord(ev_in[c], s_in), "cudaEventRecord"))
        break;
      // kernels; the output slot is free once the copy out of chunk c - 2 ran
      if (!ck(cudaStreamWaitEvent(s_comp, ev_in[c], 0), "cudaStreamWaitEvent")) break;
      if (c >= 2 && !ck(cudaStreamWaitEvent(s_comp, ev_out[c - 2], 0), "cudaStreamWaitEvent")) break;
      // the direct kernel, or the staging and attention kernels (no single
      // cooperative kernel, no cut tiles: no sync words to clear)
      ForwardPlan pl;
      st = plan_forward(device, in_ptr(c, 0), in_ptr(c, 1), in_ptr(c, 2), hn, N, D, false, 0, &pl);
      if (st == VATTN_OK)
        st = run_forward(pl, in_ptr(c, 0), in_ptr(c, 1), in_ptr(c, 2), out_ptr(c), nullptr, nullptr,
                         ws16, s_comp, device);
      if (st != VATTN_OK || !ck(cudaEventRecord(ev_comp[c], s_comp), "cudaEventRecord")) break;
      // copy out
      if (!ck(cudaStreamWaitEvent(s_out, ev_comp[c], 0), "cudaStreamWaitEvent") ||
          !ck(cudaMemcpyAsync(out + off, out_ptr(c), nb, cudaMemcpyDeviceToHost, s_out), "copy of out") ||
          !ck(cudaEventRecord(ev_out[c], s_out), "cudaEventRecord"))
        break;
    }
    // the caller's stream continues after the last copy out (which follows
    // every kernel and copy of the call); on an error, after whatever was queued
    if (st == VATTN_OK) {
      joined = ck(cudaStreamWaitEvent(stream, ev_out[n_chunks - 1], 0), "cudaStreamWaitEvent");
    }
  }
  if (!joined) {
    // make the caller's stream (and so the release below) wait for all three streams
    for (int i = 0; i < 3; ++i) {
      cudaEvent_t tail = nullptr;
      if (cudaEventCreateWithFlags(&tail, cudaEventDisableTiming) == cudaSuccess) {
        if (cudaEventRecord(tail, hs[i]) == cudaSuccess) cudaStreamWaitEvent(stream, tail, 0);
        cudaEventDestroy(tail);
      }
    }
  }
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);  // released once complete
  e = cudaFreeAsync(ws, stream);
  if (st == VATTN_OK && e != cudaSuccess) st = cuda_fail(e, "workspace release");
  return st;
}

vattn_status vattn_selftest_wait_timeout(void* stream_ptr) {
  g_last_error[0] = '\0';
  vattn_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream_ptr)>>>();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test kernel launch");
  return VATTN_OK;
}

vattn_status vattn_device_status(uint32_t* code) {
  g_last_error[0] = '\0';
  if (!code) return fail(VATTN_ERR_INVALID_ARG, "null code pointer");
  *code = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  uint32_t value = 0;
  e = cudaMemcpyFromSymbol(&value, vattn::g_vattn_status, sizeof(value));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (value != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(vattn::g_vattn_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
  }
  *code = value;
  if (value != 0)
    return fail(VATTN_ERR_DEVICE_TIMEOUT, "a kernel wait timed out (status 0x%x, site %u)", value,
                value & 0xFFu);
  return VATTN_OK;
}

const char* vattn_status_string(vattn_status status) {
  switch (status) {
    case VATTN_OK: return "VATTN_OK";
    case VATTN_ERR_INVALID_ARG: return "VATTN_ERR_INVALID_ARG";
    case VATTN_ERR_UNSUPPORTED: return "VATTN_ERR_UNSUPPORTED";
    case VATTN_ERR_MISALIGNED: return "VATTN_ERR_MISALIGNED";
    case VATTN_ERR_CUDA: return "VATTN_ERR_CUDA";
    case VATTN_ERR_DEVICE_TIMEOUT: return "VATTN_ERR_DEVICE_TIMEOUT";
  }
  return "VATTN_ERR_UNKNOWN";
}

vattn_status vattn_forward_mode_for(int64_t batch, int64_t n_heads, int64_t n_patches,
                                    int64_t head_dim, int aligned, int cooperative_launch,
                                    int blocks_per_sm, int n_sms, int* mode) {
  g_last_error[0] = '\0';
  if (!mode) return fail(VATTN_ERR_INVALID_ARG, "null mode pointer");
  *mode = VATTN_MODE_NONE;
  if (n_sms < 1) return fail(VATTN_ERR_INVALID_ARG, "n_sms must be at least 1");
  const vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  if (batch != 0 && n_heads > INT64_MAX / batch)
    return fail(VATTN_ERR_UNSUPPORTED, "batch * n_heads overflows");
  if (batch * n_heads == 0 || n_patches == 0) return VATTN_OK;
  if (n_patches > INT32_MAX || batch * n_heads > INT32_MAX)
    return fail(VATTN_ERR_UNSUPPORTED, "n_patches and batch*n_heads must fit in 32 bits");
  const bool allowed = g_single_kernel_allowed.load(std::memory_order_relaxed) != 0;
  const int N = static_cast<int>(n_patches), D = static_cast<int>(head_dim);
  *mode = forward_mode_rule(N, D, work_tiles(batch * n_heads, N, D), n_sms, aligned != 0, allowed,
                            cooperative_launch, blocks_per_sm);
  return VATTN_OK;
}

vattn_status vattn_cut_plan_for(int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, int n_blocks, int* cut) {
  g_last_error[0] = '\0';
  if (!cut) return fail(VATTN_ERR_INVALID_ARG, "null cut pointer");
  *cut = 0;
  if (n_blocks < 1) return fail(VATTN_ERR_INVALID_ARG, "n_blocks must be at least 1");
  const vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  if (batch != 0 && n_heads > INT64_MAX / batch)
    return fail(VATTN_ERR_UNSUPPORTED, "batch * n_heads overflows");
  if (batch * n_heads == 0 || n_patches == 0) return VATTN_OK;
  if (n_patches > INT32_MAX || batch * n_heads > INT32_MAX)
    return fail(VATTN_ERR_UNSUPPORTED, "n_patches and batch*n_heads must fit in 32 bits");
  const int N = static_cast<int>(n_patches);
  const int d_pad = (static_cast<int>(head_dim) + 15) & ~15;
  const int nq = query_tiles(N, d_pad);
  const long long n_tiles = batch * n_heads * ((N + vattn::kBM * nq - 1) / (vattn::kBM * nq));
  const int T = (N + vattn::kBN - 1) / vattn::kBN;
  const int grid = static_cast<int>(n_tiles < n_blocks ? n_tiles : n_blocks);
  *cut = make_schedule(n_tiles, T, grid, g_cut_allowed.load(std::memory_order_relaxed)).cut ? 1 : 0;
  return VATTN_OK;
}

vattn_status vattn_forward_mode(const float* q, const float* k, const float* v, const float* out,
                                int64_t batch, int64_t n_heads, int64_t n_patches,
                                int64_t head_dim, int* mode) {
  g_last_error[0] = '\0';
  if (!mode) return fail(VATTN_ERR_INVALID_ARG, "null mode pointer");
  *mode = VATTN_MODE_NONE;
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  int64_t bh = 0;
  bool empty = false;
  chk = check_attention_tensors(q, k, v, out, batch, n_heads, n_patches, head_dim, &bh, &empty);
  if (chk != VATTN_OK || empty) return chk;
  int device = 0;
  const cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  vattn_mode m = VATTN_MODE_NONE;
  const vattn_status st = forward_mode_on(device, q, k, v, bh, static_cast<int>(n_patches),
                                          static_cast<int>(head_dim), true, &m);
  if (st == VATTN_OK) *mode = m;
  return st;
}

int vattn_set_single_kernel(int allow) {
  return g_single_kernel_allowed.exchange(allow != 0 ? 1 : 0);
}

int vattn_set_split_tiles(int allow) {
  return g_cut_allowed.exchange(allow <= 0 ? 0 : (allow == 1 ? 1 : 2));
}

const char* vattn_last_error_string(void) { return g_last_error; }

int vattn_version(void) { return 100; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers may not allocate device memory while
// the attention runs: a plugin executed by an inference runtime that owns all
// device memory and forbids allocation inside its execute step, or a latency-
// bound loop that cannot take an allocation's cost or a late out-of-memory
// failure.  vattn_forward_noalloc serves them: its f16 staging copies of q, k
// and v live in a fixed array in the library image instead of the memory pool
// that vattn_forward draws from.
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(VATTN_NOALLOC_MAX_SCRATCH_BYTES);

// One instance per device, created when the library's device code is loaded
// on that device and kept until the process exits; every call of
// vattn_forward_noalloc on the device shares it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The second fixed array: the call's sync words (flags, cleared by a memset
// on the stream at the start of each call) and the partial results of tiles
// cut between two blocks of a balanced schedule.  A schedule whose partial
// slots do not fit (more multiprocessors than this GPU has) runs uncut.
constexpr size_t kNoAllocPartBytes = static_cast<size_t>(VATTN_NOALLOC_PART_BYTES);
static __device__ __align__(256) uint8_t g_noalloc_part[kNoAllocPartBytes];

std::mutex g_noalloc_mu;
std::atomic<void*> g_noalloc_addr[kMaxDevices];
std::atomic<void*> g_noalloc_part_addr[kMaxDevices];

// Device addresses of g_noalloc_scratch and g_noalloc_part on `device`,
// which must be current: looked up on the first call per device, then
// cached.  A failed lookup is not cached, so a later call tries again.
vattn_status noalloc_scratch(int device, uint8_t** staging, uint8_t** sync_part) {
  if (device < 0 || device >= kMaxDevices) return fail(VATTN_ERR_CUDA, "device index %d out of range", device);
  void* addr = g_noalloc_addr[device].load(std::memory_order_acquire);
  void* paddr = g_noalloc_part_addr[device].load(std::memory_order_acquire);
  if (!addr || !paddr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    addr = g_noalloc_addr[device].load(std::memory_order_relaxed);
    paddr = g_noalloc_part_addr[device].load(std::memory_order_relaxed);
    if (!addr) {
      const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the staging scratch");
      g_noalloc_addr[device].store(addr, std::memory_order_release);
    }
    if (!paddr) {
      const cudaError_t e = cudaGetSymbolAddress(&paddr, g_noalloc_part);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the partial-result scratch");
      g_noalloc_part_addr[device].store(paddr, std::memory_order_release);
    }
  }
  *staging = static_cast<uint8_t*>(addr);
  *sync_part = static_cast<uint8_t*>(paddr);
  return VATTN_OK;
}

}  // namespace

extern "C" vattn_status vattn_forward_noalloc(const float* q, const float* k, const float* v,
                                              float* out, int64_t batch, int64_t n_heads,
                                              int64_t n_patches, int64_t head_dim,
                                              void* stream_ptr) {
  g_last_error[0] = '\0';
  // ---- host-side checks (the rules of vattn_forward plus the scratch size),
  //      before any CUDA call
  vattn_status chk = check_attention_sizes(batch, n_heads, n_patches, head_dim);
  if (chk != VATTN_OK) return chk;
  int64_t bh = 0;
  bool empty = false;
  chk = check_attention_tensors(q, k, v, out, batch, n_heads, n_patches, head_dim, &bh, &empty);
  if (chk != VATTN_OK) return chk;
  if (empty) return VATTN_OK;  // nothing to compute

  const int D = static_cast<int>(head_dim);
  const int N = static_cast<int>(n_patches);
  const int d_pad = (D + 15) & ~15;
  const int64_t rows = bh * N;
  // bh * N < 2^62 / head_dim here, so these products do not overflow
  const uint64_t region = (static_cast<uint64_t>(rows) * d_pad * 2u + 255u) & ~uint64_t{255};
  if (region > kNoAllocScratchBytes / 3)
    return fail(VATTN_ERR_UNSUPPORTED,
                "problem needs %llu bytes of f16 staging scratch (3 x batch*n_heads*n_patches x "
                "round_up(head_dim, 16) x 2); vattn_forward_noalloc has %llu "
                "(VATTN_NOALLOC_MAX_SCRATCH_BYTES): call vattn_forward instead",
                (unsigned long long)(3u * region), (unsigned long long)kNoAllocScratchBytes);
  // ---- device side
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  uint8_t* ws = nullptr;
  uint8_t* wp = nullptr;
  vattn_status st = noalloc_scratch(device, &ws, &wp);
  if (st != VATTN_OK) return st;
  ForwardPlan pl;
  if ((st = plan_forward(device, q, k, v, bh, N, D, true, kNoAllocPartBytes, &pl)) != VATTN_OK)
    return st;
  // What must start at zero is cleared by the call itself: the sync words
  // (the cut tiles' arrival counts and flags, and in the single cooperative
  // kernel's mode the key-tile ready flags) sit at the start of the second
  // array and run_forward clears them with a memset on the stream (no
  // allocation).  The f16 copies of k and v are written by the attention
  // kernel in the single kernel's mode, by the staging kernel otherwise
  // (with q, every element the attention kernel reads, padding columns
  // included); each cut tile's partial is written before its flag is
  // raised.  Rows past n_patches are never read from memory (the tensor
  // maps return zeros there).  The direct f32 kernel uses no staging copy.
  return run_forward(pl, q, k, v, out, reinterpret_cast<uint32_t*>(wp),
                     reinterpret_cast<float*>(wp + pl.sync_bytes), ws,
                     static_cast<cudaStream_t>(stream_ptr), device);
}
