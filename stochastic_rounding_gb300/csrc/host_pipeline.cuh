// host_pipeline.cuh -- the host-buffer multi-tensor step: gradients copied
// in from page-locked host memory, the step, parameters copied back out,
// pipelined over chunks of consecutive tensors and three streams.
// Included by asr.cu inside its anonymous namespace (one translation unit).

// ------------------------------------------- host-buffer multi-tensor step

// A pool of CUDA events per device ordering the copy and compute streams of
// the host-buffer step.  A stream's wait on an event takes the event's state
// when the wait is queued, so an event may go back to the pool as soon as its
// record and its waits are queued.
// The pool keeps at most kEventPoolMax events per device; a call that needed
// more gives the rest back to the driver (destroying an event whose record or
// waits are still pending is deferred by CUDA until they complete).
constexpr int kEventDevices = 64;
constexpr size_t kEventPoolMax = 4096;
std::mutex g_event_mu;
std::vector<cudaEvent_t> g_event_pool[kEventDevices];

void give_events(int dev, std::vector<cudaEvent_t> &ev)
{
    std::lock_guard<std::mutex> lk(g_event_mu);
    std::vector<cudaEvent_t> &pool = g_event_pool[dev];
    for (cudaEvent_t e : ev) {
        if (pool.size() < kEventPoolMax) pool.push_back(e);
        else cudaEventDestroy(e);
    }
    ev.clear();
}

asr_status take_events(int dev, size_t count, std::vector<cudaEvent_t> &out)
{
    out.clear();
    {
        std::lock_guard<std::mutex> lk(g_event_mu);
        std::vector<cudaEvent_t> &pool = g_event_pool[dev];
        while (!pool.empty() && out.size() < count) {
            out.push_back(pool.back());
            pool.pop_back();
        }
    }
    while (out.size() < count) {
        cudaEvent_t ev;
        const cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            give_events(dev, out);
            return cuda_fail(e);
        }
        out.push_back(ev);
    }
    return ASR_OK;
}

bool page_locked(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();                  // clear the error this query may leave
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

asr_status run_adamw_host(const asr_host_tensor_desc *table, int32_t n_tensors, const asr_adamw_hparams *hp,
                          uint64_t chunk_elems, cudaStream_t stream, cudaStream_t cin, cudaStream_t cout)
{
    asr_status st = validate_hparams(hp);
    if (st != ASR_OK) return st;
    if (n_tensors < 0 || (n_tensors > 0 && !table)) return ASR_ERR_INVALID_VALUE;
    bool work = false;
    for (int32_t i = 0; i < n_tensors; ++i) {
        const asr_host_tensor_desc &h = table[i];
        st = validate_desc(h.dev);
        if (st != ASR_OK) return st;
        if (h.dev.n == 0) continue;
        work = true;
        const uintptr_t ga = h.dev.grad_dtype == ASR_BF16 ? 1 : 3, pa = h.dev.param_dtype == ASR_BF16 ? 1 : 3;
        if (!h.grad_host || (reinterpret_cast<uintptr_t>(h.grad_host) & ga) ||
            (h.param_host && (reinterpret_cast<uintptr_t>(h.param_host) & pa)))
            return ASR_ERR_INVALID_VALUE;
    }
    if (!work) return ASR_OK;
    for (int32_t i = 0; i < n_tensors; ++i) {
        const asr_host_tensor_desc &h = table[i];
        if (h.dev.n == 0) continue;
        if (!page_locked(h.grad_host) || (h.param_host && !page_locked(h.param_host))) return ASR_ERR_INVALID_VALUE;
    }
    if (chunk_elems == 0) chunk_elems = 1ull << 28;
    // chunks of consecutive tensors, [first, last)
    std::vector<std::pair<int32_t, int32_t>> chunks;
    {
        int32_t first = 0;
        uint64_t count = 0;
        for (int32_t i = 0; i < n_tensors; ++i) {
            const uint64_t n = table[i].dev.n;
            if (i > first && count + n > chunk_elems) {
                chunks.emplace_back(first, i);
                first = i;
                count = 0;
            }
            count += n;
        }
        chunks.emplace_back(first, n_tensors);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kEventDevices) return ASR_ERR_INVALID_VALUE;
    std::vector<asr_tensor_desc> descs(static_cast<size_t>(n_tensors));
    for (int32_t i = 0; i < n_tensors; ++i) descs[i] = table[i].dev;
    std::vector<cudaEvent_t> ev;
    st = take_events(dev, 2 * chunks.size() + 2, ev);
    if (st != ASR_OK) return st;
    auto fail = [&](cudaError_t err) {
        give_events(dev, ev);
        return cuda_fail(err);
    };
    // everything after the work already queued on `stream`; the steps also
    // after the copies out already queued on copy_out (an earlier call's
    // copies out read the parameters these steps overwrite)
    if ((e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cin, ev[0], 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cout, ev[0], 0)) != cudaSuccess) return fail(e);
    if ((e = cudaEventRecord(ev.back(), cout)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(stream, ev.back(), 0)) != cudaSuccess) return fail(e);
    // Copies of consecutive tensors whose host and device ranges both follow
    // on from the previous ones go out as one (the same bytes, fewer calls).
    struct Pending {
        char *dst = nullptr;
        const char *src = nullptr;
        size_t bytes = 0;
    };
    auto add = [](Pending &q, void *dst, const void *src, size_t bytes, cudaMemcpyKind kind,
                  cudaStream_t s) -> cudaError_t {
        char *d = static_cast<char *>(dst);
        const char *r = static_cast<const char *>(src);
        if (q.bytes && d == q.dst + q.bytes && r == q.src + q.bytes) {
            q.bytes += bytes;
            return cudaSuccess;
        }
        cudaError_t err = q.bytes ? cudaMemcpyAsync(q.dst, q.src, q.bytes, kind, s) : cudaSuccess;
        q.dst = d;
        q.src = r;
        q.bytes = bytes;
        return err;
    };
    auto flush = [](Pending &q, cudaMemcpyKind kind, cudaStream_t s) -> cudaError_t {
        cudaError_t err = q.bytes ? cudaMemcpyAsync(q.dst, q.src, q.bytes, kind, s) : cudaSuccess;
        q.bytes = 0;
        return err;
    };
    for (size_t c = 0; c < chunks.size(); ++c) {
        const int32_t first = chunks[c].first, last = chunks[c].second;
        Pending in;
        for (int32_t i = first; i < last; ++i) {
            const asr_host_tensor_desc &h = table[i];
            if (h.dev.n == 0) continue;
            const size_t bytes = h.dev.n * (h.dev.grad_dtype == ASR_BF16 ? 2u : 4u);
            e = add(in, const_cast<void *>(h.dev.grad), h.grad_host, bytes, cudaMemcpyHostToDevice, cin);
            if (e != cudaSuccess) return fail(e);
        }
        if ((e = flush(in, cudaMemcpyHostToDevice, cin)) != cudaSuccess) return fail(e);
        const cudaEvent_t arrived = ev[1 + 2 * c], stepped = ev[2 + 2 * c];
        if ((e = cudaEventRecord(arrived, cin)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(stream, arrived, 0)) != cudaSuccess) return fail(e);
        st = run_adamw(descs.data() + first, last - first, hp, stream);
        if (st != ASR_OK) {
            give_events(dev, ev);
            return st;
        }
        if ((e = cudaEventRecord(stepped, stream)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(cout, stepped, 0)) != cudaSuccess) return fail(e);
        Pending out;
        for (int32_t i = first; i < last; ++i) {
            const asr_host_tensor_desc &h = table[i];
            if (h.dev.n == 0 || !h.param_host) continue;
            const size_t bytes = h.dev.n * (h.dev.param_dtype == ASR_BF16 ? 2u : 4u);
            e = add(out, h.param_host, h.dev.param, bytes, cudaMemcpyDeviceToHost, cout);
            if (e != cudaSuccess) return fail(e);
        }
        if ((e = flush(out, cudaMemcpyDeviceToHost, cout)) != cudaSuccess) return fail(e);
    }
    give_events(dev, ev);
    return ASR_OK;
}
