// host_pipeline.cu -- prefill straight from host buffers, copies overlapped with compute.
//
// diffattn_fwd_host takes q, k, v and out in (pinned) host memory. The batch is cut into chunks
// of whole sequences; two chunk slots in the caller's device workspace are used in turn. Per chunk:
//   copy stream : wait until the slot's previous chunk has been computed, copy q, k, v in
//   caller stream: wait for the copies, run the prefill on the chunk (lambda formed in the kernel)
//   out stream  : wait for the prefill, copy the chunk's output back
// so chunk c + 1 is copied in while chunk c computes and chunk c - 1 is copied out. The caller's
// stream finally waits for the last copy out, so the call is asynchronous on that stream like
// every other entry point. Streams and events are created once per device and reused.
//
// When `out` is page-locked memory mapped into the device's address space (cudaHostAlloc'd or
// registered memory on a unified-address system), the prefill's epilogue stores the output rows
// straight into it over the host link: no output slot, no copy-out stream. Stores from the SMs
// share the link with the input copies better than a second copy engine does (measured on the
// GB300: 302 MB in and 101 MB out take 1.55 ms this way against 1.62 ms with two copy engines),
// and nothing is left to copy once the last piece has been computed.
//
// Causal prefills of long sequences end finer. The last sequence's keys and values stream in
// first, then its queries in pieces of rows from the last rows to the first, and each piece is
// computed as soon as its queries have landed -- its queries against the keys up to its last row
// (queries at the end of their keys: the same rows as the whole sequence's prefill, bit for bit).
// What remains after the last input has arrived is then the first rows' piece, the cheapest
// (keys up to P), instead of a whole sequence. (The earlier sequences stay whole: pieces
// throughout made the host-to-device copies, which bound the call, slower.) The pieces run on
// streams of their own, each ordered only after its own input, so they overlap one another and
// the previous sequence's compute.
#include <mutex>

#include "internal.h"

namespace da {
namespace {

constexpr int kMaxPieces = 32;
constexpr int kPieceStreams = 4;

struct DevicePipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr, piece_s[kPieceStreams] = {};
  cudaEvent_t copied[2], computed[2], drained[2], done;
  cudaEvent_t piece_in[kMaxPieces], piece_done[kMaxPieces];
  int offsets[4 * kMaxPieces];  // per piece: {0, its rows}, {0, keys received}: staged to device
};

constexpr int kMaxDevices = 64;
DevicePipe g_pipes[kMaxDevices];
std::mutex g_pipe_mutex;

cudaError_t get_pipe(DevicePipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  DevicePipe& p = g_pipes[dev];
  if (!p.ready) {
    if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (int i = 0; i < kPieceStreams; ++i)
      if ((e = cudaStreamCreateWithFlags(&p.piece_s[i], cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (int i = 0; i < 2; ++i) {
      if ((e = cudaEventCreateWithFlags(&p.copied[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.computed[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.drained[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    if ((e = cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < kMaxPieces; ++i) {
      if ((e = cudaEventCreateWithFlags(&p.piece_in[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.piece_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

}  // namespace

// Rows per piece of the last sequence, or 0 for whole-sequence chunks throughout: causal
// sequences of at least 2048 rows end in pieces of 1024 rows (a multiple of the 128-row tile; at
// most kMaxPieces - 1 pieces, larger pieces beyond that).
int host_piece_rows(int N, int flags) {
  if (!(flags & 1) || N < 2048) return 0;
  int P = 1024;
  while ((N + P - 1) / P > kMaxPieces - 1) P += 128;
  return P;
}

int host_chunk_sequences(int B, int N, int H) {
  // smallest chunk that still fills every SM about twice with CTAs (128-row tiles x heads)
  const long long per_seq = static_cast<long long>((N + 127) / 128) * H;
  long long cb = (2LL * 152 + per_seq - 1) / (per_seq > 0 ? per_seq : 1);
  if (cb < 1) cb = 1;
  if (cb > B) cb = B;
  return static_cast<int>(cb);
}

// Two slots of cb sequences' q, k, v and out (bf16), then 512 bytes for the pieces' offsets.
static size_t slot_bytes_of(int B, int N, int H, int d, int dv) {
  const int cb = host_chunk_sequences(B, N, H);
  const size_t rows = static_cast<size_t>(cb) * N * H;
  const size_t slot = rows * (2 * d + 2 * d + dv + dv) * 2;
  return (slot + 255) & ~static_cast<size_t>(255);
}

size_t host_workspace_bytes(int B, int N, int H, int d, int dv) {
  return 2 * slot_bytes_of(B, N, H, d, dv) + 4 * kMaxPieces * sizeof(int);
}

// `run` launches the prefill of one chunk (B = cb sequences) on `stream` with device pointers;
// `run_piece` that of one piece: `rows` queries (q, out) at the end of `keys` keys (k, v) of one
// sequence, with the device offset arrays {0, rows} and {0, keys}.
cudaError_t launch_host_pipeline(const HostPipeArgs& a, cudaStream_t stream,
                                 cudaError_t (*run)(const HostPipeArgs&, const void*, const void*,
                                                    const void*, void*, int, cudaStream_t, void*),
                                 cudaError_t (*run_piece)(const HostPipeArgs&, const void*,
                                                          const void*, const void*, void*, int,
                                                          int, const int*, const int*,
                                                          cudaStream_t, void*),
                                 void* ctx) {
  DevicePipe* pp = nullptr;
  cudaError_t e = get_pipe(&pp);
  if (e != cudaSuccess) return e;
  DevicePipe& p = *pp;
  // one call at a time enqueues on this device's shared copy streams and events
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  const int cb = host_chunk_sequences(a.B, a.N, a.H);
  const size_t seq_q = static_cast<size_t>(a.N) * a.H * 2 * a.d * 2;  // bytes of one sequence
  const size_t seq_v = static_cast<size_t>(a.N) * a.H * a.dv * 2;
  const size_t slot_bytes = slot_bytes_of(a.B, a.N, a.H, a.d, a.dv);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const char* qh = static_cast<const char*>(a.q);
  const char* kh = static_cast<const char*>(a.k);
  const char* vh = static_cast<const char*>(a.v);
  char* oh = static_cast<char*>(a.out);
  // the output as the kernels can address it, if the caller's buffer is mapped page-locked memory
  // (pageable memory, or page-locked memory that is not mapped: the slots and the out stream)
  char* od = nullptr;
  {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, a.out) == cudaSuccess) {
      if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr)
        od = static_cast<char*>(at.devicePointer);
    } else {
      (void)cudaGetLastError();
    }
  }
  const bool direct = od != nullptr;

  const int P = host_piece_rows(a.N, a.flags);
  const int np = P > 0 ? (a.N + P - 1) / P : 0;
  int* offs = reinterpret_cast<int*>(ws + 2 * slot_bytes);
  if (P > 0) {
    // one sequence per slot: the earlier ones as one piece of N rows (offset entry 0), the last
    // one as np pieces of P rows (entries 1 .. np; the last piece shorter)
    p.offsets[0] = 0;
    p.offsets[1] = a.N;
    p.offsets[2] = 0;
    p.offsets[3] = a.N;
    for (int i = 0; i < np; ++i) {
      const int end = (i + 1) * P < a.N ? (i + 1) * P : a.N;
      p.offsets[4 * (i + 1) + 0] = 0;
      p.offsets[4 * (i + 1) + 1] = end - i * P;
      p.offsets[4 * (i + 1) + 2] = 0;
      p.offsets[4 * (i + 1) + 3] = end;
    }
    // (from pageable memory: the call returns once the host array has been read)
    if ((e = cudaMemcpyAsync(offs, p.offsets, 4 * (np + 1) * sizeof(int), cudaMemcpyHostToDevice,
                             stream)) != cudaSuccess)
      return e;
  }
  // the slots' previous users are from an earlier call on this device: start after the caller's
  // earlier work, the offsets above included (the library's streams are non-blocking)
  if ((e = cudaEventRecord(p.done, stream)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(p.in, p.done, 0)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(p.out, p.done, 0)) != cudaSuccess) return e;
  for (int i = 0; i < (np < kPieceStreams ? np : kPieceStreams); ++i)
    if ((e = cudaStreamWaitEvent(p.piece_s[i], p.done, 0)) != cudaSuccess) return e;

  if (P > 0) {
    const size_t row_q = static_cast<size_t>(a.H) * 2 * a.d * 2, row_v = static_cast<size_t>(a.H) * a.dv * 2;
    // the sequences before the last go whole
    for (int b = 0; b < a.B - 1; ++b) {
      const int s = b & 1;
      uint8_t* dq = ws + s * slot_bytes;
      uint8_t* dk = dq + seq_q;
      uint8_t* dvv = dk + seq_q;
      uint8_t* dout = direct ? reinterpret_cast<uint8_t*>(od + b * seq_v) : dvv + seq_v;
      const size_t oq = b * seq_q, ov = b * seq_v;
      // inputs of sequence b may overwrite the slot once sequence b - 2 has been computed
      if (b >= 2 && (e = cudaStreamWaitEvent(p.in, p.computed[s], 0)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(dq, qh + oq, seq_q, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(dk, kh + oq, seq_q, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(dvv, vh + ov, seq_v, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
      if ((e = cudaEventRecord(p.copied[s], p.in)) != cudaSuccess) return e;
      // compute: its inputs are in, and the slot's output buffer was drained (sequence b - 2)
      if ((e = cudaStreamWaitEvent(stream, p.copied[s], 0)) != cudaSuccess) return e;
      if (!direct && b >= 2 && (e = cudaStreamWaitEvent(stream, p.drained[s], 0)) != cudaSuccess) return e;
      if ((e = run(a, dq, dk, dvv, dout, 1, stream, ctx)) != cudaSuccess) return e;
      if ((e = cudaEventRecord(p.computed[s], stream)) != cudaSuccess) return e;
      if (direct) continue;  // the kernel stored the rows in `out` itself
      if ((e = cudaStreamWaitEvent(p.out, p.computed[s], 0)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(oh + ov, dout, seq_v, cudaMemcpyDeviceToHost, p.out)) != cudaSuccess) return e;
      if ((e = cudaEventRecord(p.drained[s], p.out)) != cudaSuccess) return e;
    }
    // the last sequence: its keys and values first, then its queries in pieces from the last
    // rows to the first. Each piece is computed on a piece stream as soon as its queries have landed (its keys
    // are all in by then): the longest pieces start first, and the input that lands last, the
    // first rows' queries, needs the least compute (keys up to P). (Both of the last two
    // sequences as a tail, keys first, left the GPU idle while their keys streamed in: 1.77
    // against 1.68 ms at B4 N4096 H12.)
    {
      const int b = a.B - 1, s = b & 1;
      uint8_t* dq = ws + s * slot_bytes;
      uint8_t* dk = dq + seq_q;
      uint8_t* dvv = dk + seq_q;
      uint8_t* dout = direct ? reinterpret_cast<uint8_t*>(od + b * seq_v) : dvv + seq_v;
      if (b >= 2 && (e = cudaStreamWaitEvent(p.in, p.computed[s], 0)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(dk, kh + b * seq_q, seq_q, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(dvv, vh + b * seq_v, seq_v, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
      for (int j = 0; j < np; ++j) {
        const int i = np - 1 - j;               // piece i: rows i P .. i P + rows - 1
        const int e0 = 4 * (i + 1);             // its offset entry
        const int r0 = i * P, rows = p.offsets[e0 + 1];
        const size_t oq = b * seq_q + r0 * row_q, ov = b * seq_v + r0 * row_v;
        if ((e = cudaMemcpyAsync(dq + r0 * row_q, qh + oq, rows * row_q, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(p.piece_in[j], p.in)) != cudaSuccess) return e;
        // compute the piece: its queries (and so all keys) are in, and the slot's output
        // buffer was drained (sequence b - 2)
        cudaStream_t cs = p.piece_s[j % kPieceStreams];
        if ((e = cudaStreamWaitEvent(cs, p.piece_in[j], 0)) != cudaSuccess) return e;
        if (!direct && b >= 2 && (e = cudaStreamWaitEvent(cs, p.drained[s], 0)) != cudaSuccess) return e;
        if ((e = run_piece(a, dq + r0 * row_q, dk, dvv, dout + r0 * row_v, rows, r0 + rows,
                           offs + e0, offs + e0 + 2, cs, ctx)) != cudaSuccess)
          return e;
        if ((e = cudaEventRecord(p.piece_done[j], cs)) != cudaSuccess) return e;
        // the caller's stream completes after every piece
        if ((e = cudaStreamWaitEvent(stream, p.piece_done[j], 0)) != cudaSuccess) return e;
        if (direct) continue;  // the kernel stored the piece's rows in `out` itself
        if ((e = cudaStreamWaitEvent(p.out, p.piece_done[j], 0)) != cudaSuccess) return e;
        if ((e = cudaMemcpyAsync(oh + ov, dout + r0 * row_v, rows * row_v, cudaMemcpyDeviceToHost, p.out)) != cudaSuccess) return e;
      }
    }
  }

  const int chunks = P > 0 ? 0 : (a.B + cb - 1) / cb;
  for (int c = 0; c < chunks; ++c) {
    const int s = c & 1;
    const int b0 = c * cb, nb = (a.B - b0) < cb ? (a.B - b0) : cb;
    uint8_t* slot = ws + s * slot_bytes;
    uint8_t* dq = slot;
    uint8_t* dk = dq + cb * seq_q;
    uint8_t* dvv = dk + cb * seq_q;
    uint8_t* dout = direct ? reinterpret_cast<uint8_t*>(od + b0 * seq_v) : dvv + cb * seq_v;
    // inputs of chunk c may overwrite the slot once chunk c - 2 has been computed
    if (c >= 2 && (e = cudaStreamWaitEvent(p.in, p.computed[s], 0)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(dq, qh + b0 * seq_q, nb * seq_q, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(dk, kh + b0 * seq_q, nb * seq_q, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(dvv, vh + b0 * seq_v, nb * seq_v, cudaMemcpyHostToDevice, p.in)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(p.copied[s], p.in)) != cudaSuccess) return e;
    // compute: its inputs are in, and the slot's output buffer has been drained (chunk c - 2)
    if ((e = cudaStreamWaitEvent(stream, p.copied[s], 0)) != cudaSuccess) return e;
    if (!direct && c >= 2 && (e = cudaStreamWaitEvent(stream, p.drained[s], 0)) != cudaSuccess) return e;
    if ((e = run(a, dq, dk, dvv, dout, nb, stream, ctx)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(p.computed[s], stream)) != cudaSuccess) return e;
    if (direct) continue;
    // copy the chunk's output back
    if ((e = cudaStreamWaitEvent(p.out, p.computed[s], 0)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(oh + b0 * seq_v, dout, nb * seq_v, cudaMemcpyDeviceToHost, p.out)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(p.drained[s], p.out)) != cudaSuccess) return e;
  }
  // the caller's stream completes with the last copy out; the input stream is joined too so that
  // a later call cannot start copying into a slot this call still reads
  if ((e = cudaEventRecord(p.done, p.out)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(stream, p.done, 0)) != cudaSuccess) return e;
  if ((e = cudaEventRecord(p.done, p.in)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(stream, p.done, 0);
}

}  // namespace da
