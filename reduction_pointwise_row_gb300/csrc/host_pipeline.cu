// Row reductions over matrices held in host memory.  The rows travel to the
// device and back in chunks through a ring of device staging buffers, on
// three streams so that a chunk's host-to-device copy, the kernel of the
// chunk before it and the device-to-host copy of the one before that run at
// the same time (two copy directions and the SMs are independent engines;
// on GB300 the host link is NVLink-C2C).  Ordering is by events only: the
// caller's stream waits for the last copy, nothing synchronises the host.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fr.h"
#include "launch.h"

namespace fr {
namespace {

constexpr int kStageBufs = 3;  // staging slots per direction
constexpr int kMaxDev = 64;

// Streams and events of one device, created on first use and kept for the
// process (they hold no device memory of the caller's).
struct Pipe {
  bool ready = false;
  cudaStream_t h2d, comp, d2h;
  cudaEvent_t start, x_in[kStageBufs], k_done[kStageBufs], y_out[kStageBufs], end;
};

std::mutex g_pipe_mu;
Pipe g_pipe[kMaxDev];
std::mutex g_run_mu[kMaxDev];  // one caller at a time enqueues on a device's pipe

cudaError_t pipe_for(int dev, Pipe **out) {
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  Pipe &p = g_pipe[dev];
  if (!p.ready) {
    cudaError_t e;
    const unsigned sf = cudaStreamNonBlocking;
    if ((e = cudaStreamCreateWithFlags(&p.h2d, sf)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.comp, sf)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.d2h, sf)) != cudaSuccess) return e;
    const unsigned ef = cudaEventDisableTiming;
    if ((e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.end, ef)) != cudaSuccess) return e;
    for (int i = 0; i < kStageBufs; ++i) {
      if ((e = cudaEventCreateWithFlags(&p.x_in[i], ef)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.k_done[i], ef)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.y_out[i], ef)) != cudaSuccess) return e;
    }
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

}  // namespace

size_t host_pipeline_workspace(int64_t cols, int64_t esize_in, int64_t esize_out,
                               int64_t chunk_rows) {
  const size_t in = static_cast<size_t>(chunk_rows) * cols * esize_in;
  const size_t out = static_cast<size_t>(chunk_rows) * cols * esize_out;
  const size_t a_in = (in + 255) / 256 * 256, a_out = (out + 255) / 256 * 256;
  return kStageBufs * (a_in + a_out);
}

cudaError_t host_pipeline_run(const void *x_host, void *y_host, int64_t rows, int64_t cols,
                              int64_t esize_in, int64_t esize_out, int64_t chunk_rows,
                              void *workspace, cudaStream_t caller, const RowKernel &kernel) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  Pipe *p = nullptr;
  if ((e = pipe_for(dev, &p)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> run_lock(g_run_mu[dev]);
  const size_t in_bytes = static_cast<size_t>(chunk_rows) * cols * esize_in;
  const size_t out_bytes = static_cast<size_t>(chunk_rows) * cols * esize_out;
  const size_t a_in = (in_bytes + 255) / 256 * 256, a_out = (out_bytes + 255) / 256 * 256;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  auto x_dev = [&](int b) { return ws + static_cast<size_t>(b) * a_in; };
  auto y_dev = [&](int b) { return ws + kStageBufs * a_in + static_cast<size_t>(b) * a_out; };

  // everything the caller queued before this call comes first
  if ((e = cudaEventRecord(p->start, caller)) != cudaSuccess) return e;
  for (cudaStream_t s : {p->h2d, p->comp, p->d2h})
    if ((e = cudaStreamWaitEvent(s, p->start, 0)) != cudaSuccess) return e;

  const int64_t nchunks = (rows + chunk_rows - 1) / chunk_rows;
  for (int64_t i = 0; i < nchunks; ++i) {
    const int b = static_cast<int>(i % kStageBufs);
    const int64_t r0 = i * chunk_rows;
    const int64_t nr = rows - r0 < chunk_rows ? rows - r0 : chunk_rows;
    const size_t nin = static_cast<size_t>(nr) * cols * esize_in;
    const size_t nout = static_cast<size_t>(nr) * cols * esize_out;
    // slot b's input is free once the kernel of chunk i - kStageBufs is done
    if (i >= kStageBufs && (e = cudaStreamWaitEvent(p->h2d, p->k_done[b], 0)) != cudaSuccess)
      return e;
    if ((e = cudaMemcpyAsync(x_dev(b),
                             static_cast<const unsigned char *>(x_host) +
                                 static_cast<size_t>(r0) * cols * esize_in,
                             nin, cudaMemcpyHostToDevice, p->h2d)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(p->x_in[b], p->h2d)) != cudaSuccess) return e;
    // the kernel needs the chunk in, and slot b's output copied out
    if ((e = cudaStreamWaitEvent(p->comp, p->x_in[b], 0)) != cudaSuccess) return e;
    if (i >= kStageBufs && (e = cudaStreamWaitEvent(p->comp, p->y_out[b], 0)) != cudaSuccess)
      return e;
    if ((e = kernel(x_dev(b), y_dev(b), nr, p->comp)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(p->k_done[b], p->comp)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(p->d2h, p->k_done[b], 0)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(static_cast<unsigned char *>(y_host) +
                                 static_cast<size_t>(r0) * cols * esize_out,
                             y_dev(b), nout, cudaMemcpyDeviceToHost, p->d2h)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(p->y_out[b], p->d2h)) != cudaSuccess) return e;
  }
  // the caller's stream resumes after the last copy out (which follows every
  // kernel and every copy in) -- the h2d and compute streams are joined too
  if ((e = cudaEventRecord(p->end, p->h2d)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(p->d2h, p->end, 0)) != cudaSuccess) return e;
  if ((e = cudaEventRecord(p->end, p->comp)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(p->d2h, p->end, 0)) != cudaSuccess) return e;
  if ((e = cudaEventRecord(p->end, p->d2h)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(caller, p->end, 0);
}

}  // namespace fr
