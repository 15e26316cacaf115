// cc3d_writer.cu -- asynchronous chunk output: device -> pinned host -> file, overlapped with the
// next chunk's compute (the pipeline of AWS / Synthesia, "How Synthesia optimizes generative AI
// video inference on Amazon EC2 G7e instances": a copy stream beside the compute stream, double
// buffers in device and pinned host memory with events as barriers, and a worker thread that
// writes the host buffers while the main thread keeps launching kernels).
//
// Host code only.  The caller owns the device buffers (two, alternated by chunk) and the compute
// stream; the writer owns the copy stream, two pinned host slots, their events and the worker.
//   submit(n): event on the compute stream -> the copy stream waits for it -> D2H into slot n % 2
//              -> "copied" event -> the worker waits for that event, writes the slot, frees it.
//   wait_copied(n, stream): the compute stream waits for submission n's copy, before the device
//              buffer it was read from is overwritten.
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <thread>

#include <cuda_runtime.h>

#include "cc3d.h"

namespace {

constexpr int kSlots = 2;

struct Job {
    long long seq;
    int slot;
    size_t bytes;
};

}  // namespace

struct cc3d_writer_s {
    FILE* file = nullptr;
    size_t slot_bytes = 0;
    int device = -1;  // the device current at creation: its copy stream, and where src must live
    void* host[kSlots] = {nullptr, nullptr};
    cudaStream_t copy = nullptr;
    cudaEvent_t ready[kSlots] = {nullptr, nullptr};   // compute reached the submission
    cudaEvent_t copied[kSlots] = {nullptr, nullptr};  // D2H of the slot's submission done
    long long copied_seq[kSlots] = {-1, -1};          // which submission copied[slot] belongs to
    bool busy[kSlots] = {false, false};               // slot holds data not yet written
    std::mutex mu;
    std::condition_variable cv;
    std::deque<Job> queue;
    bool stop = false;
    int error = CC3D_OK;  // first failure seen by the worker
    long long next_seq = 0;
    long long bytes_written = 0;
    std::thread worker;

    void run()
    {
        for (;;) {
            Job j;
            {
                std::unique_lock<std::mutex> lock(mu);
                cv.wait(lock, [&] { return stop || !queue.empty(); });
                if (queue.empty()) return;  // stop requested and nothing left
                j = queue.front();
                queue.pop_front();
            }
            int err = CC3D_OK;
            bool failed_before;
            {
                std::lock_guard<std::mutex> lock(mu);
                failed_before = error != CC3D_OK;
            }
            // once a copy or a write has failed, the jobs queued behind it are dropped, not
            // written: the file ends at the last chunk that reached it whole, never with a gap
            // followed by later chunks
            if (cudaEventSynchronize(copied[j.slot]) != cudaSuccess) err = CC3D_ERR_CUDA;
            else if (!failed_before && j.bytes && fwrite(host[j.slot], 1, j.bytes, file) != j.bytes) err = CC3D_ERR_IO;
            {
                std::lock_guard<std::mutex> lock(mu);
                if (err != CC3D_OK && error == CC3D_OK) error = err;
                if (err == CC3D_OK && !failed_before) bytes_written += (long long)j.bytes;
                busy[j.slot] = false;
            }
            cv.notify_all();
        }
    }
};

static void writer_free(cc3d_writer_s* w)
{
    if (w == nullptr) return;
    for (int s = 0; s < kSlots; ++s) {
        if (w->host[s]) cudaFreeHost(w->host[s]);
        if (w->ready[s]) cudaEventDestroy(w->ready[s]);
        if (w->copied[s]) cudaEventDestroy(w->copied[s]);
    }
    if (w->copy) cudaStreamDestroy(w->copy);
    if (w->file) fclose(w->file);
    delete w;
}

extern "C" {

cc3d_status cc3d_writer_create(const char* path, size_t slot_bytes, cc3d_writer_t* out)
{
    if (out == nullptr) return CC3D_ERR_INVALID_ARG;
    *out = nullptr;
    if (path == nullptr || slot_bytes == 0) return CC3D_ERR_INVALID_ARG;
    cc3d_writer_s* w = new (std::nothrow) cc3d_writer_s;
    if (w == nullptr) return CC3D_ERR_OOM;
    w->slot_bytes = slot_bytes;
    w->file = fopen(path, "wb");
    if (w->file == nullptr) {
        writer_free(w);
        return CC3D_ERR_IO;
    }
    // whole slots are written at once: no stdio buffer, so a failed write leaves no part of a
    // chunk behind to be flushed later
    setvbuf(w->file, nullptr, _IONBF, 0);
    if (cudaGetDevice(&w->device) != cudaSuccess) {
        cudaGetLastError();
        writer_free(w);
        return CC3D_ERR_CUDA;
    }
    bool ok = cudaStreamCreateWithFlags(&w->copy, cudaStreamNonBlocking) == cudaSuccess;
    for (int s = 0; ok && s < kSlots; ++s) {
        ok = cudaHostAlloc(&w->host[s], slot_bytes, cudaHostAllocDefault) == cudaSuccess &&
             cudaEventCreateWithFlags(&w->ready[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&w->copied[s], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        writer_free(w);
        return CC3D_ERR_CUDA;
    }
    try {
        w->worker = std::thread([w] { w->run(); });
    } catch (...) {
        writer_free(w);
        return CC3D_ERR_OOM;
    }
    *out = w;
    return CC3D_OK;
}

cc3d_status cc3d_writer_submit(cc3d_writer_t w, const void* src, size_t bytes, void* compute_stream,
                               long long* seq_out)
{
    if (w == nullptr || src == nullptr || bytes == 0 || bytes > w->slot_bytes) return CC3D_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, src) != cudaSuccess) {
        cudaGetLastError();
        return CC3D_ERR_NOT_DEVICE_MEMORY;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return CC3D_ERR_NOT_DEVICE_MEMORY;
    if (a.type == cudaMemoryTypeDevice && a.device != w->device) return CC3D_ERR_INVALID_ARG;
    long long seq;
    int slot;
    {
        // the slot's previous contents must have reached the file
        std::unique_lock<std::mutex> lock(w->mu);
        if (w->error != CC3D_OK) return (cc3d_status)w->error;
        seq = w->next_seq;
        slot = (int)(seq % kSlots);
        w->cv.wait(lock, [&] { return !w->busy[slot] || w->error != CC3D_OK; });
        if (w->error != CC3D_OK) return (cc3d_status)w->error;
        w->busy[slot] = true;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
    if (cudaEventRecord(w->ready[slot], cs) != cudaSuccess || cudaStreamWaitEvent(w->copy, w->ready[slot], 0) != cudaSuccess ||
        cudaMemcpyAsync(w->host[slot], src, bytes, cudaMemcpyDeviceToHost, w->copy) != cudaSuccess ||
        cudaEventRecord(w->copied[slot], w->copy) != cudaSuccess) {
        std::lock_guard<std::mutex> lock(w->mu);
        w->busy[slot] = false;
        w->cv.notify_all();
        return CC3D_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lock(w->mu);
        w->copied_seq[slot] = seq;
        w->next_seq = seq + 1;
        w->queue.push_back(Job{seq, slot, bytes});
    }
    w->cv.notify_all();
    if (seq_out) *seq_out = seq;
    return CC3D_OK;
}

cc3d_status cc3d_writer_wait_copied(cc3d_writer_t w, long long seq, void* stream)
{
    if (w == nullptr) return CC3D_ERR_INVALID_ARG;
    if (seq < 0) return CC3D_OK;  // nothing submitted from that buffer yet
    const int slot = (int)(seq % kSlots);
    std::lock_guard<std::mutex> lock(w->mu);
    // the slot's event belongs to a later submission once seq + 2 has been submitted: that copy was
    // enqueued after seq's on the same copy stream, so waiting for it is waiting for seq as well
    if (seq >= w->next_seq) return CC3D_ERR_INVALID_ARG;
    if (cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), w->copied[slot], 0) != cudaSuccess) return CC3D_ERR_CUDA;
    return CC3D_OK;
}

cc3d_status cc3d_writer_close(cc3d_writer_t w, long long* bytes_written)
{
    if (w == nullptr) return CC3D_ERR_INVALID_ARG;
    {
        std::lock_guard<std::mutex> lock(w->mu);
        w->stop = true;
    }
    w->cv.notify_all();
    if (w->worker.joinable()) w->worker.join();
    int st = w->error;
    if (bytes_written) *bytes_written = w->bytes_written;
    if (fflush(w->file) != 0 && st == CC3D_OK) st = CC3D_ERR_IO;
    if (fclose(w->file) != 0 && st == CC3D_OK) st = CC3D_ERR_IO;
    w->file = nullptr;
    writer_free(w);
    return (cc3d_status)st;
}

}  // extern "C"
