// host_pipeline.cu -- attn_fwd on host buffers, with the transfers overlapped
// with the computation (the C entry point attn_fwd_host).
//
// The batch is cut into chunks of whole sequences.  Chunk c's inputs go
// host -> device on the h2d stream, its forward runs once they have arrived
// (even chunks on the caller's compute stream, odd ones on a second compute
// stream), and its outputs go device -> host on the d2h stream once the
// forward is done and every chunk's inputs are in; so the copy of chunk
// c + 1 proceeds while chunk c computes, and the read-backs run while the
// last chunks compute.  Sequences are
// independent in the forward, so every output element is the one a single
// attn_fwd call over the whole batch writes, bit for bit.
//
// A single bf16 sequence (B == 1) is cut by query rows instead.  Chunk c
// covers rows [r_c, r_c+1) (multiples of 256, the forward kernel's work
// unit) and needs keys [0, e_c): all Nk without a mask, e_c = r_c+1 + (Nk -
// Nq) with the bottom-right causal mask (Nq <= Nk), a prefix of the cache.
// The keys past the previous chunk's prefix are copied with the chunk.  The
// chunk's forward is the problem restricted to its rows: its row i (row
// r_c + i of the sequence) sees key j iff j <= i + (e_c - (r_c+1 - r_c)) =
// (r_c + i) + (Nk - Nq), the same keys as in one call over all rows, and
// every row is computed by the same arithmetic, so the results are again
// equal bit for bit.  The chunk's LSE rows are strided by Nq (one run per
// head), so they are read back with one 2-D copy.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"

namespace {

constexpr int kMaxChunks = 16;
constexpr int kRowUnit = 256;  // query rows of one work unit of the forward kernel
constexpr int kEvents = 2 * kMaxChunks + 3;

// Events the pipeline records between its streams: created on first use per
// host thread and device, then reused by every call (a recorded event may be
// recorded again once the waits on it have been enqueued).
struct EventPool {
    cudaEvent_t ev[kEvents];
    bool ready = false;
    bool get() {
        if (ready) return true;
        for (int i = 0; i < kEvents; ++i) {
            if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
                for (int k = 0; k < i; ++k) cudaEventDestroy(ev[k]);
                return false;
            }
        }
        ready = true;
        return true;
    }
    // (no destructor: the events live until the process ends, so nothing
    // calls into the CUDA runtime during its own teardown)
};

// The second compute stream: consecutive chunks' forwards run on the caller's
// stream and on this one by turns, so the next chunk's CTAs take the SMs
// that the current chunk's last wave of work units leaves idle (eight row
// chunks of one 16K-key sequence: 1.67 ms back to back on one stream, 1.56
// on two; sixteen: 1.82 and 1.52).  Created on first use per host thread and
// device, like the events; its work is ordered by events only.
struct SideStream {
    cudaStream_t s = nullptr;
    bool get() {
        return s != nullptr || cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess ||
               (s = nullptr, false);
    }
};

// Per device, so that a thread that drives several GPUs keeps one set each.
struct DeviceResources {
    EventPool events;
    SideStream side;
};
thread_local DeviceResources t_res[attn_host::kMaxDevices];

bool misaligned16(const void* p) { return (reinterpret_cast<unsigned long long>(p) & 15ull) != 0; }

}  // namespace

extern "C" attn_status_t attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                                       float* lse_h, void* q_d, void* k_d, void* v_d, void* o_d,
                                       float* lse_d, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                       int causal, float scale, attn_dtype_t dtype, int chunks,
                                       void* stream, void* h2d_stream, void* d2h_stream) {
    if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0 || Hkv < 1 || d < 1 || chunks < 0) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID;  // as attn_fwd
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0 || Nq == 0) return ATTN_OK;
    if (q_h == nullptr || o_h == nullptr || lse_h == nullptr || q_d == nullptr || o_d == nullptr ||
        lse_d == nullptr)
        return ATTN_ERR_INVALID;
    if (Nk > 0 && (k_h == nullptr || v_h == nullptr || k_d == nullptr || v_d == nullptr))
        return ATTN_ERR_INVALID;
    if (misaligned16(q_d) || misaligned16(o_d) || (Nk > 0 && (misaligned16(k_d) || misaligned16(v_d))) ||
        (reinterpret_cast<unsigned long long>(lse_d) & 3ull) != 0)
        return ATTN_ERR_INVALID;
    // One bf16 sequence: chunks of query rows (see the top of this file).
    const bool by_rows = B == 1 && dtype == ATTN_BF16 && Nk > 0 && (!causal || Nq <= Nk);
    const int row_units = (Nq + kRowUnit - 1) / kRowUnit;
    // Default: 16 row chunks for one sequence (B = 1, N = 16384 causal on
    // GB300, end to end: 1.84 ms against 1.98 with 8 and 2.29 with 12), else
    // min(B, 4).
    int n = chunks == 0 ? (by_rows ? 16 : (B < 4 ? B : 4)) : chunks;
    if (n > kMaxChunks) return ATTN_ERR_UNSUPPORTED;
    if (n > (by_rows ? row_units : B)) n = by_rows ? row_units : B;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= attn_host::kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    DeviceResources& res = t_res[dev];
    if (!res.events.get()) return ATTN_ERR_CUDA;
    if (n > 1 && !res.side.get()) return ATTN_ERR_CUDA;
    cudaEvent_t* ev = res.events.ev;
    cudaStream_t side = n > 1 ? res.side.s : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t up = h2d_stream ? static_cast<cudaStream_t>(h2d_stream) : st;
    cudaStream_t down = d2h_stream ? static_cast<cudaStream_t>(d2h_stream) : st;
    // compute stream of chunk c
    auto cstream = [&](int c) { return (c & 1) ? side : st; };
    // chunk c's inputs are in (ev_in, recorded on up after its copies); its
    // forward waits for that
    auto inputs_sent = [&](int c) -> bool {
        return up == cstream(c) || cudaEventRecord(ev[2 * c], up) == cudaSuccess;
    };
    auto wait_inputs = [&](int c) -> bool {
        cudaStream_t cs = cstream(c);
        return up == cs || cudaStreamWaitEvent(cs, ev[2 * c], 0) == cudaSuccess;
    };
    // chunk c's read-back starts once its forward is done
    auto release_outputs = [&](int c) -> bool {
        cudaStream_t cs = cstream(c);
        if (down == cs) return true;
        return cudaEventRecord(ev[2 * c + 1], cs) == cudaSuccess &&
               cudaStreamWaitEvent(down, ev[2 * c + 1], 0) == cudaSuccess;
    };

    const size_t esz = dtype == ATTN_BF16 ? 2 : 4;
    const size_t q_seq = (size_t)Nq * Hq * d * esz;    // bytes of one sequence's q (and o)
    const size_t kv_seq = (size_t)Nk * Hkv * d * esz;  // ... of its k (and v)
    const size_t l_seq = (size_t)Hq * Nq * sizeof(float);
    const char* qh = static_cast<const char*>(q_h);
    const char* kh = static_cast<const char*>(k_h);
    const char* vh = static_cast<const char*>(v_h);
    char* oh = static_cast<char*>(o_h);
    char* lh = reinterpret_cast<char*>(lse_h);
    char* qd = static_cast<char*>(q_d);
    char* kd = static_cast<char*>(k_d);
    char* vd = static_cast<char*>(v_d);
    char* od = static_cast<char*>(o_d);
    char* ld = reinterpret_cast<char*>(lse_d);

    // The read-backs start once every input copy is done: the two copy
    // directions share the host link (measured: 0.97 ms in, 0.71 ms out, 1.12
    // ms both at once), and the forwards wait for the inputs, so the inputs go
    // first (one 16K-key sequence in 16 row chunks: 1.84 ms end to end, 1.93
    // with the read-backs interleaved).
    // That pays only when the forwards outlast the read-backs: holding them
    // behind the inputs of a short computation (B = 4 x 4K keys: 0.2 ms of
    // forward for 134 MB of outputs) would serialise the two copies.  So
    // the read-backs are held when the forward's estimated time (at 1.3
    // PFLOP/s) exceeds that of the read-backs (at 190 GB/s).
    cudaEvent_t ev_all_in = ev[2 * kMaxChunks + 2];
    const double flops = 4.0 * B * Hq * (double)Nq * Nk * d * (causal ? 0.5 : 1.0);
    const double out_bytes = (double)B * (q_seq + l_seq);
    const bool hold = flops / 1.3e15 > out_bytes / 1.9e11;
    auto hold_outputs = [&]() -> bool {
        if (!hold || down == st || down == up) return true;
        return cudaEventRecord(ev_all_in, up) == cudaSuccess && cudaStreamWaitEvent(down, ev_all_in, 0) == cudaSuccess;
    };

    // the side streams start after the work already queued on the compute stream
    cudaEvent_t ev_start = ev[2 * kMaxChunks], ev_done = ev[2 * kMaxChunks + 1];
    if (cudaEventRecord(ev_start, st) != cudaSuccess) return ATTN_ERR_CUDA;
    if (up != st && cudaStreamWaitEvent(up, ev_start, 0) != cudaSuccess) return ATTN_ERR_CUDA;
    if (down != st && cudaStreamWaitEvent(down, ev_start, 0) != cudaSuccess) return ATTN_ERR_CUDA;
    if (n > 1 && cudaStreamWaitEvent(side, ev_start, 0) != cudaSuccess) return ATTN_ERR_CUDA;

    if (by_rows) {
        const size_t q_row = (size_t)Hq * d * esz;    // bytes of one query row (all heads)
        const size_t kv_row = (size_t)Hkv * d * esz;  // bytes of one key row
        long long k_done = 0;                         // keys already sent
        auto rows_of = [&](int c, int* r0, int* r1) {
            *r0 = (int)((long long)row_units * c / n) * kRowUnit;
            *r1 = c + 1 == n ? Nq : (int)((long long)row_units * (c + 1) / n) * kRowUnit;
        };
        for (int c = 0; c < n; ++c) {  // every chunk's inputs
            int r0, r1;
            rows_of(c, &r0, &r1);
            const long long k_end = causal ? (long long)r1 + (Nk - Nq) : Nk;
            if (cudaMemcpyAsync(qd + r0 * q_row, qh + r0 * q_row, (size_t)(r1 - r0) * q_row,
                                cudaMemcpyHostToDevice, up) != cudaSuccess)
                return ATTN_ERR_CUDA;
            if (k_end > k_done) {
                const size_t off = (size_t)k_done * kv_row, len = (size_t)(k_end - k_done) * kv_row;
                if (cudaMemcpyAsync(kd + off, kh + off, len, cudaMemcpyHostToDevice, up) != cudaSuccess ||
                    cudaMemcpyAsync(vd + off, vh + off, len, cudaMemcpyHostToDevice, up) != cudaSuccess)
                    return ATTN_ERR_CUDA;
                k_done = k_end;
            }
            if (!inputs_sent(c)) return ATTN_ERR_CUDA;
        }
        if (!hold_outputs()) return ATTN_ERR_CUDA;
        for (int c = 0; c < n; ++c) {  // the forwards and the read-backs
            int r0, r1;
            rows_of(c, &r0, &r1);
            const long long k_end = causal ? (long long)r1 + (Nk - Nq) : Nk;
            if (!wait_inputs(c)) return ATTN_ERR_CUDA;
            const attn_status_t s = attn_host::launch_fwd_tc(qd + r0 * q_row, kd, vd, od + r0 * q_row,
                                                             reinterpret_cast<float*>(ld) + r0, 1, Hq, Hkv,
                                                             r1 - r0, (int)k_end, d, causal, scale,
                                                             cstream(c), nullptr, Nq);
            if (s != ATTN_OK) return s;
            if (!release_outputs(c)) return ATTN_ERR_CUDA;
            if (cudaMemcpyAsync(oh + r0 * q_row, od + r0 * q_row, (size_t)(r1 - r0) * q_row,
                                cudaMemcpyDeviceToHost, down) != cudaSuccess ||
                cudaMemcpy2DAsync(lh + (size_t)r0 * sizeof(float), (size_t)Nq * sizeof(float),
                                  ld + (size_t)r0 * sizeof(float), (size_t)Nq * sizeof(float),
                                  (size_t)(r1 - r0) * sizeof(float), (size_t)Hq, cudaMemcpyDeviceToHost,
                                  down) != cudaSuccess)
                return ATTN_ERR_CUDA;
        }
    }
    if (!by_rows) {
        auto seqs_of = [&](int c, int* b0, int* b1) {
            *b0 = (int)((long long)B * c / n);
            *b1 = (int)((long long)B * (c + 1) / n);
        };
        for (int c = 0; c < n; ++c) {  // every chunk's inputs
            int b0, b1;
            seqs_of(c, &b0, &b1);
            const int nb = b1 - b0;
            if (cudaMemcpyAsync(qd + b0 * q_seq, qh + b0 * q_seq, nb * q_seq, cudaMemcpyHostToDevice, up) !=
                cudaSuccess)
                return ATTN_ERR_CUDA;
            if (Nk > 0) {
                if (cudaMemcpyAsync(kd + b0 * kv_seq, kh + b0 * kv_seq, nb * kv_seq, cudaMemcpyHostToDevice,
                                    up) != cudaSuccess ||
                    cudaMemcpyAsync(vd + b0 * kv_seq, vh + b0 * kv_seq, nb * kv_seq, cudaMemcpyHostToDevice,
                                    up) != cudaSuccess)
                    return ATTN_ERR_CUDA;
            }
            if (!inputs_sent(c)) return ATTN_ERR_CUDA;
        }
        if (!hold_outputs()) return ATTN_ERR_CUDA;
        for (int c = 0; c < n; ++c) {  // the forwards and the read-backs
            int b0, b1;
            seqs_of(c, &b0, &b1);
            const int nb = b1 - b0;
            if (!wait_inputs(c)) return ATTN_ERR_CUDA;
            const attn_status_t s = attn_fwd(qd + b0 * q_seq, Nk > 0 ? kd + b0 * kv_seq : nullptr,
                                             Nk > 0 ? vd + b0 * kv_seq : nullptr, od + b0 * q_seq,
                                             reinterpret_cast<float*>(ld + b0 * l_seq), nb, Hq, Hkv, Nq, Nk, d,
                                             causal, scale, dtype, cstream(c));
            if (s != ATTN_OK) return s;
            if (!release_outputs(c)) return ATTN_ERR_CUDA;
            if (cudaMemcpyAsync(oh + b0 * q_seq, od + b0 * q_seq, nb * q_seq, cudaMemcpyDeviceToHost, down) !=
                    cudaSuccess ||
                cudaMemcpyAsync(lh + b0 * l_seq, ld + b0 * l_seq, nb * l_seq, cudaMemcpyDeviceToHost, down) !=
                    cudaSuccess)
                return ATTN_ERR_CUDA;
        }
    }
    // the compute stream completes after the last read back
    if (down != st) {
        if (cudaEventRecord(ev_done, down) != cudaSuccess || cudaStreamWaitEvent(st, ev_done, 0) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}
