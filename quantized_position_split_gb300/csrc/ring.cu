// Step-spanning tail-prefetch ring and the native decode-step runner.
//
// Design from "Rolling-KV: step/graph-level tail prefetch (design)", section "The fix:
// a persistent, step-spanning tail-prefetch ring": B = 2..4 device staging slots sized
// once; one flat schedule of (layer, tile) tail reads per step, kept B tiles ahead on a
// dedicated copy stream; each op waits for its tile's copy_done and records
// compute_done; a slot is refilled only after its compute_done (the write-after-read
// discipline replaces a per-op barrier); events are created once, never per op.  Each
// tile is one bulk host-to-device transfer per plane, or a single transfer when its
// planes are packed in host memory as they are in the slot, after the lesson of "F5
// M7 — Rolling KV: position-windowed KV residency", section "2026-07-06 — bs2
// tail-spill curve" (one transfer per tile instead of per-head strided copies).
//
// Every wait is either a device-side stream/event dependency or a host poll with a
// deadline; nothing here can block forever.
#include <sys/mman.h>

#include <algorithm>
#include <chrono>
#include <cstring>
#include <mutex>
#include <thread>
#include <map>
#include <vector>

#include "internal.h"

namespace {
// Every allocation made by qps_host_alloc: base -> (length, made by mmap, the device's
// address of the base).  qps_host_free unregisters and unmaps the mappings (flags = 2)
// instead of calling cudaFreeHost; the ring copies a packed tile in one transfer only when
// it lies in one of them, and moves a tile with its copy kernel only when every plane does.
struct HostAlloc {
  size_t bytes;
  bool mapped;
  const char* dev;
};
std::mutex& host_map_mutex() {
  static std::mutex m;
  return m;
}
std::map<uintptr_t, HostAlloc>& host_map() {
  static std::map<uintptr_t, HostAlloc> m;
  return m;
}
// The device's address of host byte p when [p, p + n) lies inside one qps_host_alloc
// allocation, else nullptr.
const char* host_alloc_dev(const void* p, size_t n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  std::lock_guard<std::mutex> lk(host_map_mutex());
  auto it = host_map().upper_bound(a);
  if (it == host_map().begin()) return nullptr;
  --it;
  const size_t off = a - it->first;
  if (off > it->second.bytes || n > it->second.bytes - off) return nullptr;
  return it->second.dev + off;
}
bool in_one_host_alloc(const void* p, size_t n) { return host_alloc_dev(p, n) != nullptr; }

// A tile moved by the copy kernel: up to six (device-visible host source, slot offset,
// bytes) segments.
struct KernelCopy {
  const char* src[6];
  size_t off[6];
  size_t bytes[6];
  int n;
};
}  // namespace

struct qps_ring {
  static constexpr uint64_t kMagic = 0x7170735f72696e67ULL;  // "qps_ring"
  uint64_t magic = kMagic;
  int device = 0;
  int n_slots = 0;
  size_t slot_bytes = 0;
  void* alloc[4] = {nullptr, nullptr, nullptr, nullptr};  // guard + slot + guard
  void* slots[4] = {nullptr, nullptr, nullptr, nullptr};  // alloc + kGuardBytes
  cudaStream_t copy = nullptr;
  cudaEvent_t copy_done[4] = {};
  cudaEvent_t compute_done[4] = {};
  bool compute_recorded[4] = {false, false, false, false};
  std::vector<qps_tile_desc> tiles;
  std::vector<size_t> offsets;  // per tile: 6 plane offsets within the slot
  std::vector<size_t> span;     // per tile: bytes of one copy covering every plane, or 0
  std::vector<KernelCopy> kcopy;  // per tile: its copy-kernel segments (n = 0: cudaMemcpyAsync)
  int copy_mode = QPS_RING_COPY_ENGINE;
  int next_consume = 0;
  bool open = false;
  // one-shot host-side fault of the next copy of schedule index fault_tile (tests)
  int fault_tile = -1;
  int fault_mode = QPS_RING_FAULT_NONE;
  int fault_delay_ms = 0;
};

namespace qps {
namespace {

constexpr size_t kPlaneAlign = 256;
// Guard regions before and after every slot, filled with a fixed pattern at creation
// and compared by qps_ring_check_guards: a write outside its slot changes one of them.
constexpr size_t kGuardBytes = 256;
constexpr size_t kGuardWords = kGuardBytes / 4;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pattern word i of the guard before (side 0) or after (side 1) slot `slot`.
uint32_t guard_word(int slot, int side, size_t i) {
  uint32_t x = 0x9E3779B9u * (uint32_t)(i + 1) ^ (side ? 0xC0DEC0DEu : 0x5EED5EEDu) ^ (uint32_t)slot << 24;
  x ^= x >> 15;
  return x * 0x2C1B3C6Du;
}

void guard_pattern(int slot, int side, uint32_t* out) {
  for (size_t i = 0; i < kGuardWords; ++i) out[i] = guard_word(slot, side, i);
}

// Stand-in for a late tile copy: runs on the copy stream before the copy (a host
// function: it sleeps, calls no CUDA API).
void CUDART_CB late_copy_host_fn(void* ms) {
  std::this_thread::sleep_for(std::chrono::milliseconds(*static_cast<const int*>(ms)));
}

bool valid_ring(const qps_ring* r) { return r && r->magic == qps_ring::kMagic; }

qps_status check_pinned(const void* p, const char* what) {
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(QPS_ERR_INVALID_ARG, std::string(what) + ": not a CUDA-known host pointer");
  }
  if (attr.type != cudaMemoryTypeHost)
    return fail(QPS_ERR_INVALID_ARG, std::string(what) + ": tail planes must be pinned host memory");
  return QPS_OK;
}

// Host -> slot copy by SMs reading the pinned allocation through its device mapping
// (QPS_RING_COPY_KERNEL).  On some GB300 hosts the copy engine's host-to-device transfers
// stall in bursts (chunks of 1.3 ms taking up to 50 ms, seconds lost per 10 s of
// streaming); the same transfers issued as loads by SMs ran at the same 211 GB/s without
// them in every probe.
// Every segment: n16 16-byte units (source and destination 16-byte aligned), then rem
// bytes one by one.  Shape chosen inside the decode step (fp16 Qwen-like stack): 64
// CTAs of 64 threads with four 16-byte loads in flight per thread stream the tail at
// ~196 GB/s and leave each window attention at ~39 us (alone 28.6 us); pushing the copy
// to ~199 GB/s (sixteen loads in flight, or 304 x 32 threads) gains 1-2% of step time
// but slows every window launch beside it to ~95 us.
constexpr int kCopyCtas = 64, kCopyThreads = 64, kCopyUnroll = 4;

struct CopySegs {
  const uint4* src[6];
  uint4* dst[6];
  uint64_t n16[6];
  uint32_t rem[6];
  int n;
  // the slot's bytes [slot_lo, slot_hi): the checked build tests every write against them
  const uint8_t* slot_lo;
  const uint8_t* slot_hi;
  unsigned int* err;
};

__global__ void __launch_bounds__(kCopyThreads) ring_copy_kernel(const __grid_constant__ CopySegs s) {
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t step = (size_t)gridDim.x * blockDim.x;
  // a 16-byte (or, for the byte tail, one-byte) write at q stays inside the slot
  auto in_slot = [&](const void* q, size_t bytes) {
    const uint8_t* b = static_cast<const uint8_t*>(q);
    return in_bounds(b >= s.slot_lo && b + bytes <= s.slot_hi, s.err);
  };
  for (int k = 0; k < s.n; ++k) {
    const uint4* __restrict__ src = s.src[k];
    uint4* __restrict__ dst = s.dst[k];
    const size_t n = s.n16[k];
    size_t i = tid;
    for (; i + (kCopyUnroll - 1) * step < n; i += kCopyUnroll * step) {
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) v[u] = src[i + u * step];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (in_slot(dst + i + u * step, 16)) dst[i + u * step] = v[u];
    }
    for (; i < n; i += step)
      if (in_slot(dst + i, 16)) dst[i] = src[i];
    if (tid < s.rem[k] && in_slot(reinterpret_cast<uint8_t*>(dst + n) + tid, 1))
      reinterpret_cast<uint8_t*>(dst + n)[tid] = reinterpret_cast<const uint8_t*>(src + n)[tid];
  }
}

qps_status issue_copy(qps_ring* r, int i) {
  const int slot = i % r->n_slots;
  const qps_tile_desc& t = r->tiles[i];
  if (i == r->fault_tile) {  // an armed test fault: one shot
    const int mode = r->fault_mode;
    r->fault_tile = -1;
    r->fault_mode = QPS_RING_FAULT_NONE;
    if (mode == QPS_RING_FAULT_COPY_FAIL)
      return fail(QPS_ERR_CUDA, "ring: injected failure of the copy of tile " + std::to_string(i));
    if (mode == QPS_RING_FAULT_COPY_LATE)
      QPS_CUDA_TRY(cudaLaunchHostFunc(r->copy, late_copy_host_fn, &r->fault_delay_ms));
  }
  if (r->compute_recorded[slot]) QPS_CUDA_TRY(cudaStreamWaitEvent(r->copy, r->compute_done[slot], 0));
  char* base = reinterpret_cast<char*>(r->slots[slot]);
  const size_t* off = &r->offsets[(size_t)i * 6];
  if (r->kcopy[i].n > 0) {
    const KernelCopy& kc = r->kcopy[i];
    CopySegs cs{};
    cs.n = kc.n;
    cs.slot_lo = reinterpret_cast<const uint8_t*>(base);
    cs.slot_hi = reinterpret_cast<const uint8_t*>(base) + r->slot_bytes;
    cs.err = QPS_CHECK_BOUNDS ? device_error_word() : nullptr;
    for (int k = 0; k < kc.n; ++k) {
      cs.src[k] = reinterpret_cast<const uint4*>(kc.src[k]);
      cs.dst[k] = reinterpret_cast<uint4*>(base + kc.off[k]);
      cs.n16[k] = kc.bytes[k] / 16;
      cs.rem[k] = (uint32_t)(kc.bytes[k] % 16);
    }
    ring_copy_kernel<<<kCopyCtas, kCopyThreads, 0, r->copy>>>(cs);
    count_launch();
    QPS_CUDA_TRY(cudaGetLastError());
  } else if (r->span[i]) {  // the planes sit in host memory exactly as in the slot: one copy
    QPS_CUDA_TRY(cudaMemcpyAsync(base, t.host_k[0], r->span[i], cudaMemcpyHostToDevice, r->copy));
  } else {
    for (int p = 0; p < t.n_k_planes; ++p)
      if (t.bytes_k[p])
        QPS_CUDA_TRY(cudaMemcpyAsync(base + off[p], t.host_k[p], t.bytes_k[p], cudaMemcpyHostToDevice, r->copy));
    for (int p = 0; p < t.n_v_planes; ++p)
      if (t.bytes_v[p])
        QPS_CUDA_TRY(cudaMemcpyAsync(base + off[3 + p], t.host_v[p], t.bytes_v[p], cudaMemcpyHostToDevice, r->copy));
  }
  QPS_CUDA_TRY(cudaEventRecord(r->copy_done[slot], r->copy));
  return QPS_OK;
}

// Bytes a view spanning `tokens` tokens of a token-major tile needs in plane `plane`.
int64_t plane_need(const qps_kv_view& v, int plane, int d, int64_t tokens, int hkv) {
  if (tokens == 0) return 0;
  const int64_t rows = (tokens - 1) * v.tok_stride + (int64_t)(hkv - 1) * v.head_stride + 1;
  return rows * plane_row_bytes(v.fmt, plane, d);
}

qps_status tail_attend(qps_ring* r, int idx, const qps_attn_args* a_in, cudaStream_t compute,
                       int64_t parts_capacity, int* n_split_used) {
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "decode_tail: invalid or destroyed ring");
  if (!r->open) return fail(QPS_ERR_STATE, "decode_tail: no open step");
  if (!a_in) return fail(QPS_ERR_INVALID_ARG, "decode_tail: args is NULL");
  if (idx != r->next_consume)
    return fail(QPS_ERR_STATE, "decode_tail: tiles must be consumed in schedule order (expected " +
                                   std::to_string(r->next_consume) + ", got " + std::to_string(idx) + ")");
  const qps_tile_desc& t = r->tiles[idx];
  const int slot = idx % r->n_slots;
  qps_attn_args a = *a_in;
  if (a.causal) a.q_pos -= t.pos0;  // the kernel counts positions from the tile's start
  a.k.tok_stride = a.v.tok_stride = t.tok_stride;
  a.k.head_stride = a.v.head_stride = t.head_stride;
  if (t.n_k_planes != plane_count(a.k.fmt) || t.n_v_planes != plane_count(a.v.fmt))
    return fail(QPS_ERR_INVALID_ARG, "decode_tail: tile plane counts do not match the k / v formats");
  char* base = reinterpret_cast<char*>(r->slots[slot]);
  const size_t* off = &r->offsets[(size_t)idx * 6];
  const void* kp[3] = {nullptr, nullptr, nullptr};
  const void* vp[3] = {nullptr, nullptr, nullptr};
  for (int p = 0; p < t.n_k_planes; ++p) {
    kp[p] = base + off[p];
    if (plane_need(a.k, p, a.d, t.tokens, a.hkv) > (int64_t)t.bytes_k[p])
      return fail(QPS_ERR_INVALID_ARG, "decode_tail: a K plane of the tile is smaller than the view needs");
  }
  for (int p = 0; p < t.n_v_planes; ++p) {
    vp[p] = base + off[3 + p];
    if (plane_need(a.v, p, a.d, t.tokens, a.hkv) > (int64_t)t.bytes_v[p])
      return fail(QPS_ERR_INVALID_ARG, "decode_tail: a V plane of the tile is smaller than the view needs");
  }
  a.k.data = kp[0];
  a.k.aux = kp[1];
  a.k.aux2 = kp[2];
  a.v.data = vp[0];
  a.v.aux = vp[1];
  a.v.aux2 = vp[2];
  a.k.batch_stride = a.v.batch_stride = 0;  // one tail tile serves every batch entry
  a.kv_begin = 0;
  a.kv_end = t.tokens;
  AttnParams p;
  int n_split = 0;
  qps_status st = resolve_attn(&a, &p, &n_split, nullptr);
  if (st != QPS_OK) return st;
  if (a.o_parts && (int64_t)a.part_offset + n_split > parts_capacity)
    return fail(QPS_ERR_INVALID_ARG, "decode_tail: parts capacity exceeded");
  QPS_CUDA_TRY(cudaStreamWaitEvent(compute, r->copy_done[slot], 0));
  st = run_attn(&a, p, n_split, compute, parts_capacity == INT64_MAX ? -1 : parts_capacity);
  if (st != QPS_OK) return st;
  QPS_CUDA_TRY(cudaEventRecord(r->compute_done[slot], compute));
  r->compute_recorded[slot] = true;
  r->next_consume++;
  if (n_split_used) *n_split_used = n_split;
  const int next = idx + r->n_slots;
  if (next < (int)r->tiles.size()) return issue_copy(r, next);
  return QPS_OK;
}

// Side streams of the step runner: a layer with several device parts (the fan-out's
// shared prefix and private suffixes) launches its first part on the step's stream and
// the others on these, forked from and joined back to the step's stream by events.  The
// parts read independent inputs and write disjoint partial slots, so they may overlap.
// Created once per device and kept for the process; `m` serialises the fork / join
// enqueues of concurrent callers (the events are re-recorded per layer).
constexpr int kSideStreams = 3;
struct SideStreams {
  std::mutex m;
  bool ok = false;
  cudaStream_t st[kSideStreams] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kSideStreams] = {};
};
SideStreams* side_streams() {
  static std::mutex mu;
  static SideStreams* pools[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!pools[dev]) {
    SideStreams* sp = new SideStreams();
    cudaError_t e = cudaEventCreateWithFlags(&sp->fork, cudaEventDisableTiming);
    for (int i = 0; i < kSideStreams && e == cudaSuccess; ++i) {
      e = cudaStreamCreateWithFlags(&sp->st[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sp->join[i], cudaEventDisableTiming);
    }
    sp->ok = e == cudaSuccess;
    pools[dev] = sp;
  }
  return pools[dev]->ok ? pools[dev] : nullptr;
}

qps_status ring_sync(qps_ring* r, int timeout_ms) {
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
  for (;;) {
    bool busy = false;
    cudaError_t e = cudaStreamQuery(r->copy);
    if (e == cudaErrorNotReady) busy = true;
    else if (e != cudaSuccess) return cuda_fail(e, "ring_sync: cudaStreamQuery");
    for (int s = 0; s < r->n_slots && !busy; ++s) {
      if (!r->compute_recorded[s]) continue;
      e = cudaEventQuery(r->compute_done[s]);
      if (e == cudaErrorNotReady) busy = true;
      else if (e != cudaSuccess) return cuda_fail(e, "ring_sync: cudaEventQuery");
    }
    if (!busy) return QPS_OK;
    if (std::chrono::steady_clock::now() >= deadline)
      return fail(QPS_ERR_TIMEOUT, "ring_sync: copies or tail attention still running at the deadline");
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

}  // namespace
}  // namespace qps

using namespace qps;

extern "C" {

qps_status qps_host_alloc(size_t bytes, int32_t flags, void** out) {
  if (!out) return fail(QPS_ERR_INVALID_ARG, "host_alloc: out is NULL");
  *out = nullptr;
  if (bytes == 0) return fail(QPS_ERR_INVALID_ARG, "host_alloc: bytes must be > 0");
  if (flags < 0 || flags > 2) return fail(QPS_ERR_INVALID_ARG, "host_alloc: flags must be 0, 1 or 2");
  if (flags == 2) {
    // anonymous mapping advised to use transparent huge pages, faulted in, then
    // page-locked and registered with CUDA: fewer, larger pages for the copy engine
    const size_t align = (size_t)2 << 20;
    const size_t n = (bytes + align - 1) / align * align;
    void* p = mmap(nullptr, n, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (p == MAP_FAILED) return fail(QPS_ERR_CUDA, "host_alloc: mmap failed");
    madvise(p, n, MADV_HUGEPAGE);
    std::memset(p, 0, n);
    cudaError_t e = cudaHostRegister(p, n, cudaHostRegisterPortable | cudaHostRegisterMapped);
    if (e != cudaSuccess) {
      munmap(p, n);
      return cuda_fail(e, "host_alloc: cudaHostRegister");
    }
    void* dev = nullptr;
    e = cudaHostGetDevicePointer(&dev, p, 0);
    if (e != cudaSuccess) {
      cudaHostUnregister(p);
      munmap(p, n);
      return cuda_fail(e, "host_alloc: cudaHostGetDevicePointer");
    }
    std::lock_guard<std::mutex> lk(host_map_mutex());
    host_map()[reinterpret_cast<uintptr_t>(p)] = HostAlloc{n, true, reinterpret_cast<const char*>(dev)};
    *out = p;
    return QPS_OK;
  }
  unsigned int f = cudaHostAllocPortable | cudaHostAllocMapped | (flags == 1 ? cudaHostAllocWriteCombined : 0u);
  QPS_CUDA_TRY(cudaHostAlloc(out, bytes, f));
  void* dev = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(&dev, *out, 0);
  if (e != cudaSuccess) {
    cudaFreeHost(*out);
    *out = nullptr;
    return cuda_fail(e, "host_alloc: cudaHostGetDevicePointer");
  }
  std::lock_guard<std::mutex> lk(host_map_mutex());
  host_map()[reinterpret_cast<uintptr_t>(*out)] = HostAlloc{bytes, false, reinterpret_cast<const char*>(dev)};
  return QPS_OK;
}

qps_status qps_host_free(void* p) {
  if (!p) return QPS_OK;
  size_t mapped = 0;
  {
    std::lock_guard<std::mutex> lk(host_map_mutex());
    auto it = host_map().find(reinterpret_cast<uintptr_t>(p));
    if (it != host_map().end()) {
      if (it->second.mapped) mapped = it->second.bytes;
      host_map().erase(it);
    }
  }
  if (mapped) {
    QPS_CUDA_TRY(cudaHostUnregister(p));
    munmap(p, mapped);
    return QPS_OK;
  }
  QPS_CUDA_TRY(cudaFreeHost(p));
  return QPS_OK;
}

qps_status qps_ring_create(int32_t n_slots, size_t slot_bytes, int32_t device, qps_ring** out) {
  if (!out) return fail(QPS_ERR_INVALID_ARG, "ring_create: out is NULL");
  *out = nullptr;
  if (n_slots < 2 || n_slots > 4) return fail(QPS_ERR_INVALID_ARG, "ring_create: n_slots must be 2..4");
  if (slot_bytes == 0) return fail(QPS_ERR_INVALID_ARG, "ring_create: slot_bytes must be > 0");
  if (device < 0) return fail(QPS_ERR_INVALID_ARG, "ring_create: device must be >= 0");
  QPS_CUDA_TRY(cudaSetDevice(device));
  qps_ring* r = new qps_ring();
  r->device = device;
  r->n_slots = n_slots;
  r->slot_bytes = align_up(slot_bytes, kPlaneAlign);
  qps_status st = QPS_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking);
  // The copy kernel needs no shared memory; asking for the largest shared carveout keeps
  // an SM that runs one of its CTAs configured for the attention CTAs beside it (with
  // the default an SM could pick an L1-heavy split and turn the attention CTAs away)
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ring_copy_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  for (int s = 0; s < n_slots && e == cudaSuccess; ++s) {
    e = cudaMalloc(&r->alloc[s], kGuardBytes + r->slot_bytes + kGuardBytes);
    if (e == cudaSuccess) {
      r->slots[s] = static_cast<char*>(r->alloc[s]) + kGuardBytes;
      uint32_t pat[kGuardWords];
      guard_pattern(s, 0, pat);
      e = cudaMemcpy(r->alloc[s], pat, kGuardBytes, cudaMemcpyHostToDevice);
      guard_pattern(s, 1, pat);
      if (e == cudaSuccess)
        e = cudaMemcpy(static_cast<char*>(r->slots[s]) + r->slot_bytes, pat, kGuardBytes, cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->copy_done[s], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->compute_done[s], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    st = cuda_fail(e, "ring_create");
    for (int s = 0; s < 4; ++s) {
      if (r->alloc[s]) cudaFree(r->alloc[s]);
      if (r->copy_done[s]) cudaEventDestroy(r->copy_done[s]);
      if (r->compute_done[s]) cudaEventDestroy(r->compute_done[s]);
    }
    if (r->copy) cudaStreamDestroy(r->copy);
    r->magic = 0;
    delete r;
    return st;
  }
  *out = r;
  return QPS_OK;
}

qps_status qps_ring_destroy(qps_ring* r) {
  if (!r) return QPS_OK;
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_destroy: invalid or destroyed ring");
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(r->device);
  qps_status st = ring_sync(r, 10000);
  if (st != QPS_OK) {
    cudaSetDevice(prev);
    return st;
  }
  for (int s = 0; s < r->n_slots; ++s) {
    cudaFree(r->alloc[s]);
    cudaEventDestroy(r->copy_done[s]);
    cudaEventDestroy(r->compute_done[s]);
  }
  cudaStreamDestroy(r->copy);
  r->magic = 0;
  delete r;
  cudaSetDevice(prev);
  return QPS_OK;
}

qps_status qps_ring_set_copy_mode(qps_ring* r, int32_t mode) {
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_set_copy_mode: invalid or destroyed ring");
  if (mode != QPS_RING_COPY_ENGINE && mode != QPS_RING_COPY_KERNEL)
    return fail(QPS_ERR_INVALID_ARG, "ring_set_copy_mode: unknown mode");
  if (r->open) return fail(QPS_ERR_STATE, "ring_set_copy_mode: a step is open");
  r->copy_mode = mode;
  return QPS_OK;
}

qps_status qps_ring_begin_step(qps_ring* r, const qps_tile_desc* tiles, int32_t n_tiles,
                               void* compute_stream) {
  (void)compute_stream;
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_begin_step: invalid or destroyed ring");
  if (r->open) return fail(QPS_ERR_STATE, "ring_begin_step: the previous step is still open");
  if (n_tiles < 0 || (n_tiles > 0 && !tiles)) return fail(QPS_ERR_INVALID_ARG, "ring_begin_step: bad tile list");
  std::vector<size_t> offsets((size_t)n_tiles * 6, 0), span((size_t)n_tiles, 0);
  std::vector<KernelCopy> kcopy((size_t)n_tiles);
  for (int i = 0; i < n_tiles; ++i) {
    const qps_tile_desc& t = tiles[i];
    if (t.n_k_planes < 1 || t.n_k_planes > 3 || t.n_v_planes < 1 || t.n_v_planes > 3 || t.tokens < 0)
      return fail(QPS_ERR_INVALID_ARG, "ring_begin_step: tile " + std::to_string(i) + " has bad plane counts or tokens");
    if (t.tok_stride <= 0 || t.head_stride < 0)
      return fail(QPS_ERR_INVALID_ARG, "ring_begin_step: tile " + std::to_string(i) + " has bad strides");
    size_t cur = 0;
    for (int p = 0; p < 6; ++p) {
      const bool is_k = p < 3;
      const int pi = is_k ? p : p - 3;
      if (pi >= (is_k ? t.n_k_planes : t.n_v_planes)) continue;
      const void* h = is_k ? t.host_k[pi] : t.host_v[pi];
      const size_t b = is_k ? t.bytes_k[pi] : t.bytes_v[pi];
      if (b > 0) {
        if (!h) return fail(QPS_ERR_INVALID_ARG, "ring_begin_step: NULL host plane");
        qps_status st = check_pinned(h, "ring_begin_step");
        if (st != QPS_OK) return st;
      }
      offsets[(size_t)i * 6 + p] = cur;
      cur = align_up(cur + b, kPlaneAlign);
    }
    if (cur > r->slot_bytes)
      return fail(QPS_ERR_INVALID_ARG, "ring_begin_step: tile " + std::to_string(i) + " does not fit in a slot");
    // one copy suffices when every plane starts at its slot offset from the first
    // plane's host address (the tail packed tile by tile, planes 256-byte aligned) and
    // the whole span lies in one allocation of this library (a copy may not cross
    // separately pinned ranges)
    bool contiguous = t.bytes_k[0] > 0;
    size_t end = 0;
    const char* h0 = reinterpret_cast<const char*>(t.host_k[0]);
    for (int p = 0; p < 6 && contiguous; ++p) {
      const bool is_k = p < 3;
      const int pi = is_k ? p : p - 3;
      if (pi >= (is_k ? t.n_k_planes : t.n_v_planes)) continue;
      const char* h = reinterpret_cast<const char*>(is_k ? t.host_k[pi] : t.host_v[pi]);
      const size_t b = is_k ? t.bytes_k[pi] : t.bytes_v[pi];
      if (b == 0) continue;
      contiguous = h >= h0 && (size_t)(h - h0) == offsets[(size_t)i * 6 + p];
      end = offsets[(size_t)i * 6 + p] + b;
    }
    span[i] = contiguous && in_one_host_alloc(h0, end) ? end : 0;
    // the copy kernel takes the tile when every segment lies in a qps_host_alloc
    // allocation and starts on a 16-byte boundary (slot offsets are 256-byte aligned)
    KernelCopy kc{};
    bool ok = true;
    auto add = [&](const void* h, size_t off, size_t b) {
      if (!ok || b == 0) return;
      const char* dev = host_alloc_dev(h, b);
      if (!dev || (reinterpret_cast<uintptr_t>(dev) & 15)) {
        ok = false;
        return;
      }
      kc.src[kc.n] = dev;
      kc.off[kc.n] = off;
      kc.bytes[kc.n] = b;
      ++kc.n;
    };
    if (span[i]) {
      add(h0, 0, span[i]);
    } else {
      for (int p = 0; p < t.n_k_planes; ++p) add(t.host_k[p], offsets[(size_t)i * 6 + p], t.bytes_k[p]);
      for (int p = 0; p < t.n_v_planes; ++p) add(t.host_v[p], offsets[(size_t)i * 6 + 3 + p], t.bytes_v[p]);
    }
    if (!ok || r->copy_mode != QPS_RING_COPY_KERNEL) kc.n = 0;
    kcopy[i] = kc;
  }
  int prev = 0;
  cudaGetDevice(&prev);
  if (prev != r->device) return fail(QPS_ERR_INVALID_ARG, "ring_begin_step: the ring's device is not current");
  r->tiles.assign(tiles, tiles + n_tiles);
  r->offsets.swap(offsets);
  r->span.swap(span);
  r->kcopy.swap(kcopy);
  r->next_consume = 0;
  r->open = true;
  const int first = n_tiles < r->n_slots ? n_tiles : r->n_slots;
  for (int i = 0; i < first; ++i) {
    qps_status st = issue_copy(r, i);
    if (st != QPS_OK) {
      r->open = false;
      return st;
    }
  }
  return QPS_OK;
}

qps_status qps_attn_decode_tail(qps_ring* r, int32_t tile_index, const qps_attn_args* a,
                                void* compute_stream) {
  return tail_attend(r, tile_index, a, reinterpret_cast<cudaStream_t>(compute_stream), INT64_MAX,
                     nullptr);
}

qps_status qps_ring_end_step(qps_ring* r) {
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_end_step: invalid or destroyed ring");
  if (!r->open) return fail(QPS_ERR_STATE, "ring_end_step: no open step");
  if (r->next_consume != (int)r->tiles.size()) {
    r->open = false;
    return fail(QPS_ERR_STATE, "ring_end_step: " + std::to_string(r->tiles.size() - r->next_consume) +
                                   " tiles were never consumed");
  }
  r->open = false;
  return QPS_OK;
}

qps_status qps_ring_sync(qps_ring* r, int32_t timeout_ms) {
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_sync: invalid or destroyed ring");
  if (timeout_ms < 0) return fail(QPS_ERR_INVALID_ARG, "ring_sync: timeout_ms must be >= 0");
  return ring_sync(r, timeout_ms);
}

qps_status qps_ring_check_guards(qps_ring* r, int32_t timeout_ms, int32_t* bad_slot) {
  if (bad_slot) *bad_slot = -1;
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_check_guards: invalid or destroyed ring");
  if (timeout_ms < 0) return fail(QPS_ERR_INVALID_ARG, "ring_check_guards: timeout_ms must be >= 0");
  int prev = 0;
  cudaGetDevice(&prev);
  if (prev != r->device) return fail(QPS_ERR_INVALID_ARG, "ring_check_guards: the ring's device is not current");
  qps_status st = ring_sync(r, timeout_ms);  // every writer of the slots (the copies) is done
  if (st != QPS_OK) return st;
  uint32_t got[kGuardWords], want[kGuardWords];
  for (int s = 0; s < r->n_slots; ++s) {
    for (int side = 0; side < 2; ++side) {
      const char* g = side ? static_cast<const char*>(r->slots[s]) + r->slot_bytes : static_cast<const char*>(r->alloc[s]);
      QPS_CUDA_TRY(cudaMemcpy(got, g, kGuardBytes, cudaMemcpyDeviceToHost));
      guard_pattern(s, side, want);
      if (std::memcmp(got, want, kGuardBytes) != 0) {
        if (bad_slot) *bad_slot = s;
        return fail(QPS_ERR_INTERNAL, "ring_check_guards: the guard " + std::string(side ? "after" : "before") +
                                          " slot " + std::to_string(s) + " was overwritten");
      }
    }
  }
  return QPS_OK;
}

qps_status qps_ring_slot(qps_ring* r, int32_t slot, void** data, size_t* bytes) {
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_slot: invalid or destroyed ring");
  if (slot < 0 || slot >= r->n_slots) return fail(QPS_ERR_INVALID_ARG, "ring_slot: slot out of range");
  if (data) *data = r->slots[slot];
  if (bytes) *bytes = r->slot_bytes;
  return QPS_OK;
}

qps_status qps_ring_inject_fault(qps_ring* r, int32_t tile_index, int32_t mode, int32_t delay_ms) {
  if (!valid_ring(r)) return fail(QPS_ERR_STATE, "ring_inject_fault: invalid or destroyed ring");
  if (mode != QPS_RING_FAULT_NONE && mode != QPS_RING_FAULT_COPY_FAIL && mode != QPS_RING_FAULT_COPY_LATE)
    return fail(QPS_ERR_INVALID_ARG, "ring_inject_fault: unknown mode");
  if (tile_index < 0) return fail(QPS_ERR_INVALID_ARG, "ring_inject_fault: tile_index must be >= 0");
  if (mode == QPS_RING_FAULT_COPY_LATE && (delay_ms < 0 || delay_ms > 5000))
    return fail(QPS_ERR_INVALID_ARG, "ring_inject_fault: delay_ms must be in [0, 5000]");
  r->fault_tile = mode == QPS_RING_FAULT_NONE ? -1 : tile_index;
  r->fault_mode = mode;
  r->fault_delay_ms = delay_ms;
  return QPS_OK;
}

qps_status qps_copy_host(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return QPS_OK;
  if (!dst || !src) return fail(QPS_ERR_INVALID_ARG, "copy_host: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15)
    return fail(QPS_ERR_INVALID_ARG, "copy_host: dst and src must be 16-byte aligned");
  const char* src_dev = host_alloc_dev(src, bytes);
  const char* dst_dev = host_alloc_dev(dst, bytes);
  if ((src_dev != nullptr) == (dst_dev != nullptr))
    return fail(QPS_ERR_INVALID_ARG,
                "copy_host: exactly one of dst / src must lie (whole) inside qps_host_alloc memory");
  // the other side must be device memory: a plain host pointer there would be a wild
  // address for the kernel
  cudaPointerAttributes attr{};
  const void* dev_side = src_dev ? dst : src;
  if (cudaPointerGetAttributes(&attr, dev_side) != cudaSuccess ||
      (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)) {
    cudaGetLastError();  // clear a sticky error of the query itself
    return fail(QPS_ERR_INVALID_ARG, "copy_host: the side not in qps_host_alloc memory must be device memory");
  }
  uint8_t* d = dst_dev ? reinterpret_cast<uint8_t*>(const_cast<char*>(dst_dev)) : static_cast<uint8_t*>(dst);
  const uint8_t* sp = src_dev ? reinterpret_cast<const uint8_t*>(src_dev) : static_cast<const uint8_t*>(src);
  CopySegs cs{};
  cs.n = 1;
  cs.src[0] = reinterpret_cast<const uint4*>(sp);
  cs.dst[0] = reinterpret_cast<uint4*>(d);
  cs.n16[0] = bytes / 16;
  cs.rem[0] = (uint32_t)(bytes % 16);
  cs.slot_lo = d;
  cs.slot_hi = d + bytes;
  cs.err = QPS_CHECK_BOUNDS ? device_error_word() : nullptr;
  // as many CTAs as the copy has 4-vector rounds of one CTA, at most the ring's 64
  const size_t per_cta = (size_t)kCopyThreads * kCopyUnroll;
  const int ctas = (int)std::min<size_t>(kCopyCtas, std::max<size_t>(1, (cs.n16[0] + per_cta - 1) / per_cta));
  ring_copy_kernel<<<ctas, kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(cs);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

qps_status qps_decode_step(qps_ring* ring, const qps_tile_desc* tiles, int32_t n_tiles,
                           const qps_layer_step* layers, int32_t n_layers, void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n_layers < 0 || (n_layers > 0 && !layers)) return fail(QPS_ERR_INVALID_ARG, "decode_step: bad layer list");
  int64_t want_tiles = 0;
  for (int l = 0; l < n_layers; ++l) {
    if (layers[l].n_tiles < 0 || layers[l].n_device_parts < 0)
      return fail(QPS_ERR_INVALID_ARG, "decode_step: negative part or tile count");
    if (layers[l].n_tiles > 0 && !layers[l].tail) return fail(QPS_ERR_INVALID_ARG, "decode_step: tail template missing");
    if (layers[l].n_device_parts + layers[l].n_tiles == 0)
      return fail(QPS_ERR_INVALID_ARG, "decode_step: a layer has no parts");
    want_tiles += layers[l].n_tiles;
  }
  if (want_tiles != n_tiles) return fail(QPS_ERR_INVALID_ARG, "decode_step: tile count does not match the layers' n_tiles");
  if (n_tiles > 0 && !ring) return fail(QPS_ERR_INVALID_ARG, "decode_step: tiles given without a ring");
  if (ring) {
    qps_status st = qps_ring_begin_step(ring, tiles, n_tiles, stream);
    if (st != QPS_OK) return st;
  }
  qps_status st = QPS_OK;
  int tile = 0;
  for (int l = 0; l < n_layers && st == QPS_OK; ++l) {
    const qps_layer_step& L = layers[l];
    int off = 0;
    int64_t rows = -1;
    int d = 0;
    if (L.part_events[0]) {
      cudaError_t e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(L.part_events[0]), s);
      if (e != cudaSuccess) st = cuda_fail(e, "decode_step: cudaEventRecord");
    }
    // the device parts: every one resolved first (its partial slots follow the previous
    // part's), then the first launched on the step's stream and the others on side
    // streams forked from it and joined back before the layer's tiles
    std::vector<qps_attn_args> pa;
    std::vector<AttnParams> pp;
    std::vector<int> pn;
    for (int i = 0; i < L.n_device_parts && st == QPS_OK; ++i) {
      qps_attn_args a = L.device_parts[i];
      a.o_parts = L.o_parts;
      a.lse_parts = L.lse_parts;
      a.part_offset = off;
      AttnParams p;
      int n = 0;
      st = resolve_attn(&a, &p, &n, nullptr);
      if (st != QPS_OK) break;
      if (off + n > L.parts_capacity) {
        st = fail(QPS_ERR_INVALID_ARG, "decode_step: parts_capacity exceeded in layer " + std::to_string(l));
        break;
      }
      rows = p.rows_total;
      d = p.d;
      pa.push_back(a);
      pp.push_back(p);
      pn.push_back(n);
      off += n;
    }
    if (st == QPS_OK && !pa.empty()) {
      SideStreams* side = pa.size() > 1 ? side_streams() : nullptr;
      std::unique_lock<std::mutex> lk;
      int used = 0;  // side streams forked in this layer
      if (side) {
        lk = std::unique_lock<std::mutex>(side->m);
        cudaError_t e = cudaEventRecord(side->fork, s);
        if (e != cudaSuccess) st = cuda_fail(e, "decode_step: cudaEventRecord");
      }
      for (size_t i = 0; i < pa.size() && st == QPS_OK; ++i) {
        cudaStream_t si = s;
        if (side && i > 0) {
          const int k = (int)((i - 1) % kSideStreams);
          si = side->st[k];
          if (k >= used) {
            cudaError_t e = cudaStreamWaitEvent(si, side->fork, 0);
            if (e != cudaSuccess) {
              st = cuda_fail(e, "decode_step: cudaStreamWaitEvent");
              break;
            }
            used = k + 1;
          }
        }
        st = run_attn(&pa[i], pp[i], pn[i], si, L.parts_capacity);
      }
      // join every forked stream, also after an error, so that nothing enqueued on the
      // step's stream afterwards can overtake a part still running beside it
      for (int k = 0; k < used; ++k) {
        cudaError_t e = cudaEventRecord(side->join[k], side->st[k]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, side->join[k], 0);
        if (e != cudaSuccess && st == QPS_OK) st = cuda_fail(e, "decode_step: joining a side stream");
      }
    }
    if (st == QPS_OK && L.part_events[1]) {
      cudaError_t e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(L.part_events[1]), s);
      if (e != cudaSuccess) st = cuda_fail(e, "decode_step: cudaEventRecord");
    }
    for (int j = 0; j < L.n_tiles && st == QPS_OK; ++j, ++tile) {
      qps_attn_args a = *L.tail;
      a.o_parts = L.o_parts;
      a.lse_parts = L.lse_parts;
      a.part_offset = off;
      int used = 0;
      st = tail_attend(ring, tile, &a, s, L.parts_capacity, &used);
      if (st != QPS_OK) break;
      rows = (int64_t)a.batch * (a.n_q > 1 ? a.n_q : 1) * a.hq;
      d = a.d;
      off += used;
    }
    if (st != QPS_OK) break;
    if (!L.o || !L.lse) {
      st = fail(QPS_ERR_INVALID_ARG, "decode_step: o / lse are NULL");
      break;
    }
    st = launch_combine(L.o_parts, L.lse_parts, off, rows, d, L.o, L.lse, s, device_error_word());
  }
  if (ring) {
    if (st != QPS_OK) {
      ring->open = false;
      return st;
    }
    return qps_ring_end_step(ring);
  }
  return st;
}

}  // extern "C"
