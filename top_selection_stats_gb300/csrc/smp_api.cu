// smp_api.cu -- host side of the C ABI declared in include/smp.h: argument
// checks, launch planning (cluster size, slice length, shared memory) and the
// sigma-truncation table.  All work is enqueued on the caller's stream; no
// call allocates, copies to the host or synchronises.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/smp.h"
#include "smp_core.cuh"
#include "smp_split.cuh"

namespace smp {
const void* kernel_f32();
const void* kernel_bf16();
const void* kernel_f16();
cudaError_t launch_f32(const KArgs& a, int grid, cudaStream_t st);
cudaError_t launch_bf16(const KArgs& a, int grid, cudaStream_t st);
cudaError_t launch_f16(const KArgs& a, int grid, cudaStream_t st);
const void* split_kernel_bf16();
const void* split_kernel_f16();
cudaError_t split_launch_bf16(const XArgs& a, int smem, cudaStream_t st);
cudaError_t split_launch_f16(const XArgs& a, int smem, cudaStream_t st);
int verify_enqueue(const float* p, const float* q, const int32_t* d, int B, int G, int V,
                   int64_t ld, const uint64_t* seed, const uint64_t* offset, int32_t* out_tokens,
                   int32_t* n_acc, int32_t* status, cudaStream_t st);
cudaError_t penalty_setup();
int toplp_enqueue(const void* logits, int dtype, int B, int V, long long ld, const uint32_t* kept,
                  const float* temperature, const int32_t* tokens, const float* logprobs, int n,
                  int32_t* out_ids, float* out_lp, cudaStream_t st);
int gumbel_enqueue(const void* logits, int dtype, int B, int V, long long ld,
                   const uint32_t* kept, const float* temperature, const uint64_t* seed,
                   const uint64_t* offset, int32_t* tokens, int32_t* status, cudaStream_t st);
int penalty_enqueue(void* logits, int dtype, int B, int V, long long ld, const int32_t* history,
                    int H, long long hld, const float* penalty, int32_t* status,
                    cudaStream_t st);
}  // namespace smp

using namespace smp;

struct smp_ctx {
  int device;
  int max_batch, max_vocab;
  int sm_count;
  int smem_optin;
  int smem_per_sm;
  int grid_max;
  float delta[DTAB];
  int32_t* row_info;
  int kernel;    // SMP_KERNEL_BOARD or SMP_KERNEL_SPLIT
  long long wait_limit;  // SM clock cycles a bounded device wait may take
  Board* board;  // job board: zeroed at creation, reset by each launch's last CTA
};

namespace {

// Upper-tail normal quantile: z with 0.5 * erfc(z / sqrt 2) = q, by bisection
// (Qrita paper notes, "training strategy": delta = Phi^-1(1 - k/V)).
double upper_quantile(double q) {
  if (q >= 1.0) return -8.0;
  double lo = -8.0, hi = 8.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    const double tail = 0.5 * std::erfc(mid / std::sqrt(2.0));
    if (tail > q) lo = mid;
    else hi = mid;
  }
  return 0.5 * (lo + hi);
}

const void* kernel_for(int dt) {
  switch (dt) {
    case DT_F32: return kernel_f32();
    case DT_BF16: return kernel_bf16();
    default: return kernel_f16();
  }
}

int chunk_elems(int dt) { return STAGE_BYTES / esize_of(dt); }

// Split-row launch plan (bf16 / fp16): the smallest power-of-two cluster
// (at most XMAXC CTAs) that gives the launch at least two CTAs per SM, so that
// every row streams at once; slices of at most XMAXST stages, each a multiple
// of 256 values; no CTA without values.  Rows too long for XMAXC slices take
// the streaming kernel instead (returns false).
struct XPlan {
  int C, SL, wf, cap, smem;
};
constexpr int XSMEM_MAX = (XNS * XSB + 4096 * 2 + 8192 * 2 + 8192 * 4) + (int)sizeof(XSh);
bool split_plan(int dt, int B, int V, int sms, XPlan* out) {
  if (dt != DT_BF16 && dt != DT_F16) return false;
  const long long smax = (long long)XMAXST * XVS * 8;  // values per slice, at most
  int C = 1;
  while (C < XMAXC && ((long long)B * C < 2LL * sms || (V + C - 1) / C > smax)) C *= 2;
  while (C > 1 && (long long)(C - 1) * 256 >= V) C /= 2;  // every CTA holds values
  const int SL = ((V + C - 1) / C + 255) / 256 * 256;
  if (SL > smax) return false;
  out->C = C;
  out->SL = SL;
  out->wf = dt == DT_F16 ? 4096 : 2048;
  out->cap = C >= 2 ? 2048 : 8192;
  out->smem = xoff_sh(out->wf, out->cap) + (int)sizeof(XSh);
  return true;
}
cudaError_t split_setup() {
  for (const void* k : {split_kernel_bf16(), split_kernel_f16()}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, XSMEM_MAX);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
constexpr long long WAIT_LIMIT = 4000000000ll;  // about two seconds of SM clock

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

int launch(smp_ctx* h, int mode, const void* logits, int dt, int B, int V, int64_t ld,
           const uint32_t* bitmask, const smp_row_params* params, int32_t* tokens,
           int32_t* status, uint32_t* kept_mask, int32_t* kept_count, float* probs,
           smp_stream stream, float* logprob = nullptr) {
  if (!h || !logits || !status) return SMP_ERR_INVALID_PARAM;
  if (dt != DT_F32 && dt != DT_BF16 && dt != DT_F16) return SMP_ERR_INVALID_PARAM;
  if (B < 0 || V < 1 || ld < V) return SMP_ERR_INVALID_PARAM;
  if (mode != MODE_ARGMAX &&
      (!params || !params->temperature || !params->top_k || !params->top_p))
    return SMP_ERR_INVALID_PARAM;
  if (mode == MODE_SAMPLE && (!params->seed || !params->offset || !tokens))
    return SMP_ERR_INVALID_PARAM;
  if (mode == MODE_MASK && (!kept_mask || !kept_count)) return SMP_ERR_INVALID_PARAM;
  if (mode == MODE_ARGMAX && !tokens) return SMP_ERR_INVALID_PARAM;
  if (B > h->max_batch || V > h->max_vocab) return SMP_ERR_CAPACITY;
  if ((long long)V > (long long)MAXCH * chunk_elems(dt)) return SMP_ERR_CAPACITY;
  if (B == 0) return SMP_OK;
  DeviceGuard guard(h->device);

  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.logits = logits;
  a.ld = ld;
  a.B = B;
  a.V = V;
  a.W = (V + 31) / 32;
  a.bitmask = bitmask;
  if (params) {
    a.temperature = params->temperature;
    a.top_k = params->top_k;
    a.top_p = params->top_p;
    a.seed = reinterpret_cast<const unsigned long long*>(params->seed);
    a.offset = reinterpret_cast<const unsigned long long*>(params->offset);
  }
  a.tokens = tokens;
  a.status = status;
  a.kept_mask = kept_mask;
  a.kept_count = kept_count;
  a.probs = probs;
  a.logprob = logprob;
  a.row_info = h->row_info;
  a.board = h->board;
  a.mode = mode;
  const size_t es = (size_t)esize_of(dt);
  a.use_tma = ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && ((size_t)ld * es) % 16 == 0) ? 1 : 0;
  std::memcpy(a.delta, h->delta, sizeof(a.delta));
  a.wait_limit = h->wait_limit;

  XPlan xp;
  if (h->kernel == SMP_KERNEL_SPLIT && split_plan(dt, B, V, h->sm_count, &xp)) {
    XArgs r;
    std::memset(&r, 0, sizeof(r));
    r.logits = logits;
    r.ld = ld;
    r.B = B;
    r.V = V;
    r.W = a.W;
    r.bitmask = bitmask;
    r.temperature = a.temperature;
    r.top_k = a.top_k;
    r.top_p = a.top_p;
    r.seed = a.seed;
    r.offset = a.offset;
    r.tokens = tokens;
    r.status = status;
    r.kept_mask = kept_mask;
    r.kept_count = kept_count;
    r.probs = probs;
    r.logprob = logprob;
    r.row_info = h->row_info;
    r.mode = mode;
    r.C = xp.C;
    r.SL = xp.SL;
    r.wf = xp.wf;
    r.cap = xp.cap;
    r.aligned = a.use_tma;
    r.wait_limit = h->wait_limit;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = dt == DT_BF16 ? split_launch_bf16(r, xp.smem, st)
                                        : split_launch_f16(r, xp.smem, st);
    return e == cudaSuccess ? SMP_OK : SMP_ERR_CUDA;
  }

  // one CTA per row, at most two resident per SM; CTAs loop over rows.  With
  // a job board and rows long enough to share (jobs are published for rows
  // of three chunks or more) the whole resident grid is launched: CTAs
  // without a row take chunk tasks of the slow rows from the start.
  const int nch = (V + chunk_elems(dt) - 1) / chunk_elems(dt);
  const bool helpers = h->board && nch > 2;
  const int grid = (B < h->grid_max && !helpers) ? B : h->grid_max;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (dt) {
    case DT_F32: e = launch_f32(a, grid, st); break;
    case DT_BF16: e = launch_bf16(a, grid, st); break;
    default: e = launch_f16(a, grid, st); break;
  }
  if (e != cudaSuccess) return SMP_ERR_CUDA;
  return SMP_OK;
}

}  // namespace

extern "C" {

int smp_create(smp_handle* out, int device, int max_batch, int max_vocab) {
  if (!out || max_batch < 1 || max_vocab < 1) return SMP_ERR_INVALID_PARAM;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return SMP_ERR_CUDA;
  }
  DeviceGuard guard(device);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return SMP_ERR_CUDA;
  smp_ctx* h = new smp_ctx();
  h->device = device;
  h->max_batch = max_batch;
  h->max_vocab = max_vocab;
  h->sm_count = prop.multiProcessorCount;
  h->smem_optin = (int)prop.sharedMemPerBlockOptin;
  h->smem_per_sm = (int)prop.sharedMemPerMultiprocessor;
  h->row_info = nullptr;
  h->kernel = SMP_KERNEL_BOARD;
  h->wait_limit = WAIT_LIMIT;
  for (int i = 0; i < DTAB; ++i) {
    const double l2q = -24.0 + 0.25 * i;
    h->delta[i] = (float)upper_quantile(std::pow(2.0, l2q));
  }
  const void* ks[3] = {kernel_for(DT_F32), kernel_for(DT_BF16), kernel_for(DT_F16)};
  int per_sm = 1 << 30;
  for (const void* k : ks) {
    int nb = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, NT, SMEM_TOTAL) != cudaSuccess) {
      cudaGetLastError();
      delete h;
      return SMP_ERR_CUDA;
    }
    per_sm = nb < per_sm ? nb : per_sm;
  }
  if (per_sm < 1 || penalty_setup() != cudaSuccess || split_setup() != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return SMP_ERR_CUDA;
  }
  h->grid_max = per_sm * h->sm_count;
  h->board = nullptr;
  if (cudaMalloc(&h->board, sizeof(Board)) != cudaSuccess ||
      cudaMemset(h->board, 0, sizeof(Board)) != cudaSuccess) {
    cudaGetLastError();
    if (h->board) cudaFree(h->board);
    delete h;
    return SMP_ERR_CUDA;
  }
  *out = h;
  return SMP_OK;
}

int smp_destroy(smp_handle h) {
  if (h) {
    DeviceGuard guard(h->device);
    if (h->board) cudaFree(h->board);
  }
  delete h;
  return SMP_OK;
}

int smp_topk_topp_mask(smp_handle h, const void* logits, smp_dtype dtype, int B, int V,
                       int64_t ld, const uint32_t* bitmask, const smp_row_params* params,
                       uint32_t* kept_mask, int32_t* kept_count, int32_t* row_status,
                       float* probs_out, smp_stream stream) {
  return launch(h, MODE_MASK, logits, (int)dtype, B, V, ld, bitmask, params, nullptr,
                row_status, kept_mask, kept_count, probs_out, stream);
}

int smp_sample(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
               const uint32_t* bitmask, const smp_row_params* params, int32_t* tokens,
               int32_t* row_status, uint32_t* kept_mask, int32_t* kept_count,
               smp_stream stream) {
  return launch(h, MODE_SAMPLE, logits, (int)dtype, B, V, ld, bitmask, params, tokens,
                row_status, kept_mask, kept_count, nullptr, stream);
}

int smp_sample_logprob(smp_handle h, const void* logits, smp_dtype dtype, int B, int V,
                       int64_t ld, const uint32_t* bitmask, const smp_row_params* params,
                       int32_t* tokens, float* logprobs, int32_t* row_status,
                       uint32_t* kept_mask, int32_t* kept_count, smp_stream stream) {
  if (!logprobs) return SMP_ERR_INVALID_PARAM;
  return launch(h, MODE_SAMPLE, logits, (int)dtype, B, V, ld, bitmask, params, tokens,
                row_status, kept_mask, kept_count, nullptr, stream, logprobs);
}

int smp_argmax(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
               const uint32_t* bitmask, int32_t* tokens, int32_t* row_status,
               smp_stream stream) {
  return launch(h, MODE_ARGMAX, logits, (int)dtype, B, V, ld, bitmask, nullptr, tokens,
                row_status, nullptr, nullptr, nullptr, stream);
}

int smp_set_row_info(smp_handle h, int32_t* row_info) {
  if (!h) return SMP_ERR_INVALID_PARAM;
  h->row_info = row_info;
  return SMP_OK;
}

int smp_set_kernel(smp_handle h, int kernel) {
  if (!h || (kernel != SMP_KERNEL_BOARD && kernel != SMP_KERNEL_SPLIT)) return SMP_ERR_INVALID_PARAM;
  h->kernel = kernel;
  return SMP_OK;
}

int smp_set_wait_limit(smp_handle h, long long cycles) {
  if (!h) return SMP_ERR_INVALID_PARAM;
  h->wait_limit = cycles > 0 ? cycles : WAIT_LIMIT;
  return SMP_OK;
}

int smp_plan(smp_handle h, smp_dtype dtype, int B, int V, int* cluster, int* slice,
             int* smem_bytes, int* capacity) {
  if (!h || V < 1 || B < 1) return SMP_ERR_INVALID_PARAM;
  if ((int)dtype < 0 || (int)dtype > 2) return SMP_ERR_INVALID_PARAM;
  XPlan xp;
  if (h->kernel == SMP_KERNEL_SPLIT && split_plan((int)dtype, B, V, h->sm_count, &xp)) {
    if (cluster) *cluster = xp.C;
    if (slice) *slice = xp.SL;
    if (smem_bytes) *smem_bytes = xp.smem;
    if (capacity) *capacity = xp.cap;
    return SMP_OK;
  }
  const int ce = chunk_elems((int)dtype);
  if (cluster) *cluster = 1;
  if (slice) *slice = ce;
  if (smem_bytes) *smem_bytes = SMEM_TOTAL;
  if (capacity) *capacity = CAP;
  return ((long long)V > (long long)MAXCH * ce) ? SMP_ERR_CAPACITY : SMP_OK;
}

int smp_spec_verify(smp_handle h, const float* target_probs, const float* draft_probs,
                    const int32_t* draft_tokens, int B, int G, int V, int64_t ld,
                    const uint64_t* seed, const uint64_t* offset, int32_t* out_tokens,
                    int32_t* n_accepted, int32_t* row_status, smp_stream stream) {
  if (!h || B < 0 || G < 0 || V < 1 || ld < V || (ld & 3)) return SMP_ERR_INVALID_PARAM;
  if (B == 0) return SMP_OK;
  if (!target_probs || !seed || !offset || !out_tokens || !n_accepted || !row_status)
    return SMP_ERR_INVALID_PARAM;
  if (G > 0 && (!draft_probs || !draft_tokens)) return SMP_ERR_INVALID_PARAM;
  if ((reinterpret_cast<uintptr_t>(target_probs) & 15) ||
      (G > 0 && (reinterpret_cast<uintptr_t>(draft_probs) & 15)))
    return SMP_ERR_INVALID_PARAM;
  if (B > h->max_batch || V > h->max_vocab) return SMP_ERR_CAPACITY;
  DeviceGuard guard(h->device);
  return verify_enqueue(target_probs, draft_probs, draft_tokens, B, G, V, ld, seed, offset,
                        out_tokens, n_accepted, row_status, (cudaStream_t)stream);
}

int smp_repetition_penalty(smp_handle h, void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                           const int32_t* history, int H, int64_t history_ld,
                           const float* penalty, int32_t* row_status, smp_stream stream) {
  if (!h || !logits || !penalty || !row_status) return SMP_ERR_INVALID_PARAM;
  if ((int)dtype < 0 || (int)dtype > 2) return SMP_ERR_INVALID_PARAM;
  if (B < 0 || V < 1 || ld < V || H < 0 || history_ld < H) return SMP_ERR_INVALID_PARAM;
  if (H > 0 && !history) return SMP_ERR_INVALID_PARAM;
  if (B > h->max_batch || V > h->max_vocab) return SMP_ERR_CAPACITY;
  DeviceGuard guard(h->device);
  return penalty_enqueue(logits, (int)dtype, B, V, ld, history, H, history_ld, penalty,
                         row_status, (cudaStream_t)stream);
}

int smp_gumbel_sample(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                      const uint32_t* kept_mask, const float* temperature, const uint64_t* seed,
                      const uint64_t* offset, int32_t* tokens, int32_t* row_status,
                      smp_stream stream) {
  if (!h || !logits || !temperature || !seed || !offset || !tokens || !row_status)
    return SMP_ERR_INVALID_PARAM;
  if ((int)dtype < 0 || (int)dtype > 2) return SMP_ERR_INVALID_PARAM;
  if (B < 0 || V < 1 || ld < V) return SMP_ERR_INVALID_PARAM;
  if (B > h->max_batch || V > h->max_vocab) return SMP_ERR_CAPACITY;
  DeviceGuard guard(h->device);
  return gumbel_enqueue(logits, (int)dtype, B, V, ld, kept_mask, temperature, seed, offset, tokens,
                        row_status, (cudaStream_t)stream);
}

int smp_top_logprobs(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                     const uint32_t* kept_mask, const float* temperature, const int32_t* tokens,
                     const float* logprobs, int n, int32_t* top_ids, float* top_logprobs,
                     smp_stream stream) {
  if (!h || !logits || !kept_mask || !temperature || !tokens || !logprobs || !top_ids ||
      !top_logprobs)
    return SMP_ERR_INVALID_PARAM;
  if ((int)dtype < 0 || (int)dtype > 2) return SMP_ERR_INVALID_PARAM;
  if (B < 0 || V < 1 || ld < V || n < 1) return SMP_ERR_INVALID_PARAM;
  if (B > h->max_batch || V > h->max_vocab) return SMP_ERR_CAPACITY;
  DeviceGuard guard(h->device);
  return toplp_enqueue(logits, (int)dtype, B, V, ld, kept_mask, temperature, tokens, logprobs, n,
                       top_ids, top_logprobs, (cudaStream_t)stream);
}

const char* smp_status_string(int code) {
  switch (code) {
    case SMP_OK: return "ok";
    case SMP_ERR_EMPTY: return "empty candidate set";
    case SMP_ERR_NONFINITE: return "NaN or +inf in a legal slot";
    case SMP_ERR_INVALID_PARAM: return "invalid parameter";
    case SMP_ERR_TIMEOUT: return "bounded device wait expired";
    case SMP_ERR_CUDA: return "CUDA error";
    case SMP_ERR_CAPACITY: return "beyond capacity";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// smp_sample_noalloc: the sampling call without a handle, for callers that may
// not allocate device memory.  Its only scratch is the job board (the handle
// calls take theirs from the handle's workspace); here it is the file-scope
// array below, which the CUDA runtime places on every device that loads this
// library and keeps until the process exits.  On the host the array's name
// denotes a host-side shadow object, not device memory, so the per-device
// set-up asks the runtime for its device address and passes that to the
// kernel.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t NOALLOC_SCRATCH_BYTES = (sizeof(Board) + 255) / 256 * 256;
static_assert(NOALLOC_SCRATCH_BYTES == 1968896, "the scratch size is stated in smp.h");
constexpr int NOALLOC_MAX_DEVICES = 64;
}  // namespace

static __device__ __align__(256) unsigned char smp_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex noalloc_mutex;
smp_ctx noalloc_dev[NOALLOC_MAX_DEVICES];
bool noalloc_ready[NOALLOC_MAX_DEVICES];

// Once per device context, with that device current: the kernels' shared-
// memory attribute and the resident grid (as smp_create computes them), the
// sigma table, the scratch's device address, and a clear of the scratch on
// the caller's stream.  The board must start at zero; every launch's last CTA
// leaves it at zero again, so later calls need no clear of their own.  Each
// call asks for the scratch's address again: after a device reset (a new
// primary context) the array moves, and the set-up is redone.
int noalloc_setup(int dev, cudaStream_t st, smp_ctx** out) {
  std::lock_guard<std::mutex> lock(noalloc_mutex);
  smp_ctx& c = noalloc_dev[dev];
  if (noalloc_ready[dev]) {
    void* now = nullptr;
    if (cudaGetSymbolAddress(&now, smp_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return SMP_ERR_CUDA;
    }
    if (now != (void*)c.board) noalloc_ready[dev] = false;
  }
  if (!noalloc_ready[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return SMP_ERR_CUDA;
    }
    int per_sm = 1 << 30;
    for (int dt : {DT_F32, DT_BF16, DT_F16}) {
      const void* k = kernel_for(dt);
      int nb = 0;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, NT, SMEM_TOTAL) != cudaSuccess) {
        cudaGetLastError();
        return SMP_ERR_CUDA;
      }
      per_sm = nb < per_sm ? nb : per_sm;
    }
    if (per_sm < 1) return SMP_ERR_CUDA;
    if (split_setup() != cudaSuccess) {
      cudaGetLastError();
      return SMP_ERR_CUDA;
    }
    Board* board = nullptr;
    if (cudaGetSymbolAddress((void**)&board, smp_noalloc_scratch) != cudaSuccess ||
        cudaMemsetAsync(board, 0, NOALLOC_SCRATCH_BYTES, st) != cudaSuccess) {
      cudaGetLastError();
      return SMP_ERR_CUDA;
    }
    c.device = dev;
    c.max_batch = INT_MAX;
    c.max_vocab = INT_MAX;
    c.sm_count = prop.multiProcessorCount;
    c.smem_optin = (int)prop.sharedMemPerBlockOptin;
    c.smem_per_sm = (int)prop.sharedMemPerMultiprocessor;
    c.grid_max = per_sm * c.sm_count;
    for (int i = 0; i < DTAB; ++i) c.delta[i] = (float)upper_quantile(std::pow(2.0, -24.0 + 0.25 * i));
    c.row_info = nullptr;
    c.kernel = SMP_KERNEL_BOARD;
    c.wait_limit = WAIT_LIMIT;
    c.board = board;
    noalloc_ready[dev] = true;
  }
  *out = &c;
  return SMP_OK;
}

}  // namespace

extern "C" int smp_sample_noalloc(const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                                  const uint32_t* bitmask, const smp_row_params* params,
                                  int32_t* tokens, int32_t* row_status, uint32_t* kept_mask,
                                  int32_t* kept_count, smp_stream stream) {
  const int dt = (int)dtype;
  if (!logits || !params || !tokens || !row_status) return SMP_ERR_INVALID_PARAM;
  if (dt != DT_F32 && dt != DT_BF16 && dt != DT_F16) return SMP_ERR_INVALID_PARAM;
  if (B < 0 || V < 1 || ld < V) return SMP_ERR_INVALID_PARAM;
  // the board's per-job chunk-mass table covers MAXCH staging chunks of a row
  if ((long long)V > (long long)MAXCH * chunk_elems(dt)) return SMP_ERR_CAPACITY;
  if (B == 0) return SMP_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SMP_ERR_CUDA;
  }
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return SMP_ERR_CAPACITY;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  smp_ctx* c = nullptr;
  const int rc = noalloc_setup(dev, st, &c);
  if (rc != SMP_OK) return rc;
  return launch(c, MODE_SAMPLE, logits, dt, B, V, ld, bitmask, params, tokens, row_status,
                kept_mask, kept_count, nullptr, stream);
}
