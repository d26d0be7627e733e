// Greedy token and softmax confidence from logits the caller already has, without allocating.
//
// Who needs this: code that cannot call cudaMalloc on its request path, for example a serving
// engine that hands all device memory to its own pool before the first request (so a new
// allocation fails), or a plugin running inside a host process that forbids the library from
// allocating (cudaMalloc may also synchronise the device and stall every other stream). Such a
// caller cannot provide the workspace that dflash_create needs, but it can still turn a block of
// logits -- for instance the target's own verify logits -- into greedy tokens and confidences.
//
// The reduction is the one the LM-head epilogue uses (per-CTA online max / sum of exp / lowest
// index, then the last CTA of each row merges the partials in CTA order); its scratch lives in
// g_noalloc_scratch below instead of a caller workspace.
#include <mutex>

#include "common.cuh"

namespace {

using dfl::warp_sum;

constexpr int kRowsMax = DFLASH_NOALLOC_MAX_ROWS;
constexpr int kCtasPerRow = 64;
constexpr int kThreads = 256;

struct Scratch {
  float part[kRowsMax][kCtasPerRow][3];   // per (row, CTA): max, sum of exp, index bits
  int ticket[kRowsMax];                   // CTAs of the row that have finished
};

// Every device that loads the library holds this array until the process exits (~49 KB).
static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(Scratch)];

struct St {
  float m, s;
  int i;
};

__device__ __forceinline__ void merge(St& a, const St& b) {
  if (b.m > a.m || (b.m == a.m && b.i < a.i)) {
    a.s = (a.m == -INFINITY) ? b.s : b.s + a.s * __expf(a.m - b.m);
    a.m = b.m;
    a.i = b.i;
  } else if (b.m != -INFINITY) {
    a.s += b.s * __expf(b.m - a.m);
  }
}

__global__ void __launch_bounds__(kThreads) greedy_from_logits_kernel(const float* __restrict__ logits, int vocab,
                                                                      int32_t* token, float* conf, Scratch* sc) {
  const int row = blockIdx.y, c = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long b0 = (long long)c * vocab / kCtasPerRow, b1 = (long long)(c + 1) * vocab / kCtasPerRow;
  const float* lr = logits + (size_t)row * vocab;
  St st{-INFINITY, 0.f, 0x7fffffff};
  for (long long j = b0 + threadIdx.x; j < b1; j += kThreads) {
    const float v = lr[j];
    if (v > st.m) {
      st.s = (st.m == -INFINITY) ? 1.f : st.s * __expf(st.m - v) + 1.f;
      st.m = v;
      st.i = (int)j;
    } else if (v != -INFINITY) {   // a -inf logit is masked out: it adds nothing to the sum
      st.s += __expf(v - st.m);
    }
  }
  for (int o = 1; o < 32; o <<= 1) {
    St ot{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.s, o),
          __shfl_xor_sync(0xffffffffu, st.i, o)};
    merge(st, ot);
  }
  __shared__ St sw[kThreads / 32];
  __shared__ int last;
  if (lane == 0) sw[warp] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    St acc = sw[0];
    for (int w = 1; w < kThreads / 32; w++) merge(acc, sw[w]);
    sc->part[row][c][0] = acc.m;
    sc->part[row][c][1] = acc.s;
    sc->part[row][c][2] = __int_as_float(acc.i);
    __threadfence();
    last = atomicAdd(&sc->ticket[row], 1) == kCtasPerRow - 1;
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  St acc{-INFINITY, 0.f, 0x7fffffff};
  for (int k = 0; k < kCtasPerRow; k++) {
    St o{__ldcg(&sc->part[row][k][0]), __ldcg(&sc->part[row][k][1]), __float_as_int(__ldcg(&sc->part[row][k][2]))};
    merge(acc, o);
  }
  // a row whose every logit is -inf has no greedy token
  const bool none = acc.m == -INFINITY;
  token[row] = none ? -1 : acc.i;
  if (conf) conf[row] = none ? 0.f : 1.0f / acc.s;
  sc->ticket[row] = 0;
}

// Device address of g_noalloc_scratch per device ordinal, looked up once with that device current.
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(Scratch** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DFLASH_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DFLASH_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<Scratch*>(g_scratch_ptr[dev]);
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_greedy_from_logits_noalloc(const float* logits, int rows, int vocab, int32_t* token,
                                                 float* conf, void* stream) {
  if (rows == 0) return DFLASH_OK;
  if (!logits || !token || rows < 0 || vocab < 2) return DFLASH_EINVAL;
  if (rows > kRowsMax) return DFLASH_ECAPACITY;
  Scratch* sc = nullptr;
  const int st = scratch_for_current_device(&sc);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the tickets must start at zero; the partials are always written before they are read
  if (cudaMemsetAsync(sc->ticket, 0, sizeof(int) * rows, s) != cudaSuccess) return DFLASH_ECUDA;
  greedy_from_logits_kernel<<<dim3(kCtasPerRow, rows), kThreads, 0, s>>>(logits, vocab, token, conf, sc);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ECUDA;
}
