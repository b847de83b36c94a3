"""Training-time activation offload through the ZVC path.

Rhu et al., "Compressing DMA Engine", section V.D: vDNN moves the activation maps that a
layer's backward pass will need out of GPU memory during forward propagation and brings
them back ahead of the backward pass; cDMA compresses them on the way. `ActivationOffload`
does this for any PyTorch model through autograd's saved-tensor hooks:

    off = ActivationOffload(where="host")
    with off:
        loss = model(x).sum()
    loss.backward()

pack (forward): every saved CUDA tensor of a 4-byte dtype with at least `min_elems`
    elements, other than a parameter, is compressed with zvc_offload into pinned host
    memory (where="host"), or with zvc_compress into a device buffer of exactly the
    compressed size (where="device": the compressed stream stays in HBM, the paper's
    future-work use). Autograd then keeps the handle, not the tensor. A tensor saved by
    several operators (a ReLU output is saved by the ReLU and by the next layer) is
    compressed once. zvc_offload waits on the host for each segment's compressed size, so
    in host mode it runs on a worker thread: the training loop's thread only records an
    event and queues the tensor, and keeps enqueueing the forward pass.
unpack (backward): the tensor is restored bit for bit (zvc_prefetch or zvc_decompress) on a
    side stream. Tensors are unpacked in about the reverse order of packing, so restoring
    tensor k also starts restoring the tensor packed just before it, overlapping the
    backward work in between; that tensor's unpack then only waits for its event.

All compression and restoration runs in this package's CUDA kernels; this module only
allocates buffers and orders streams. The compressed copy of a tensor is released when
autograd drops its handle (after the backward pass unless the graph is retained); a pinned
buffer goes back to the allocator only once the device is done with it.
"""
from __future__ import annotations

import collections
import queue
import threading
import weakref

from . import (ZVC_DEFAULT_CHUNK_ELEMS, ZvcError, _check, get_error, new_workspace,
               zvc_compress, zvc_decompress, zvc_offload, zvc_offload_host_bound,
               zvc_offload_join, zvc_offload_workspace_size, zvc_prefetch, zvc_size_bound,
               zvc_workspace_size)


def _torch():
    import torch
    return torch


def _offload_worker(owner_ref, jobs):
    """Worker thread of one ActivationOffload: offloads its queued tensors in order. It
    holds the offloader only while a job runs, and ends on None or once the offloader is
    gone."""
    while True:
        job = jobs.get()
        if job is None:
            return
        h, t, produced, cap = job
        job = None
        owner = owner_ref()
        try:
            if owner is None:
                raise RuntimeError("ActivationOffload dropped before its tensors were offloaded")
            owner._offload_one(h, t, produced, cap)
        except BaseException as e:  # reported on the training loop's thread
            h.error = e
        finally:
            t = owner = None
            h.offloaded.set()
            h = None


class _Packed:
    """A saved tensor in compressed form."""
    __slots__ = ("shape", "dtype", "device", "n", "host", "size", "dev", "order", "peers",
                 "saves", "unpacks", "out", "ready", "done", "owner", "offloaded", "error",
                 "__weakref__")

    def __init__(self, t, order, peers, owner):
        self.shape, self.dtype, self.device = t.shape, t.dtype, t.device
        self.n = t.numel()
        self.host = self.dev = self.out = self.ready = self.done = None
        self.size = 0
        self.order = order    # position in its forward pass
        self.peers = peers    # weak references to that pass's handles, in pack order
        self.saves = 1        # operators that saved this tensor
        self.unpacks = 0
        self.owner = owner    # weak reference to the ActivationOffload
        self.offloaded = None  # host mode: set once the worker has offloaded the tensor
        self.error = None      # host mode: the worker's exception, if any

    def __del__(self):
        owner = self.owner() if self.owner is not None else None
        if owner is not None and self.host is not None:
            # the device may still read or write the pinned buffer until `done`
            with owner._lock:
                owner._retired.append((self.host, self.done))


class ActivationOffload:
    """Saved-tensor hooks that keep activations ZVC-compressed between forward and backward.

    where: "host" (pinned host memory, through zvc_offload/zvc_prefetch) or "device"
        (compressed stream kept in HBM, through zvc_compress/zvc_decompress).
    min_elems: smaller tensors are kept as they are.
    prefetch_ahead: on unpack of tensor k, start restoring the tensor packed before it.
    max_pending: host mode: tensors queued for the worker but not yet offloaded, at most;
        the training loop waits beyond that. A queued tensor still occupies its device
        memory, so this bounds what the offload costs in memory while the loop runs ahead.
        (On the deep CNN of `bench.py --train`: 0, 1, 2, 4, 8 give 45.2, 42.5, 43.2, 43.3,
        44.7 ms per step at 2.48, 2.48, 2.48, 2.87, 4.51 GB of peak extra memory.)
    """

    def __init__(self, where: str = "host", min_elems: int = 1 << 16,
                 chunk_elems: int = ZVC_DEFAULT_CHUNK_ELEMS, prefetch_ahead: bool = True,
                 max_pending: int = 1):
        if where not in ("host", "device"):
            raise ValueError(where)
        self.where, self.min_elems, self.C = where, int(min_elems), int(chunk_elems)
        self.prefetch_ahead = prefetch_ahead
        self._lock = threading.RLock()  # also taken by handles dropped on the worker thread
        self._ws = {}        # device -> workspace tensor (grown on demand)
        self._keep = []      # replaced workspaces: the copy stream may still use them
        self._retired = []   # (pinned buffer, event): dropped once the event has completed
        self._side = {}      # device -> side stream for restores
        self._join = {}      # device -> stream that joins the offload copies
        self._seen = {}      # address of a saved tensor -> (tensor weakref, handle), this pass
        self._order = []     # this forward pass's handles (weak references), in pack order
        self._hooks = None
        self._jobs = None     # host mode: queue of the worker thread
        self._worker = None
        self._wstream = {}    # device -> stream the worker compresses on
        self.max_pending = max(0, int(max_pending))
        self._pending = collections.deque()  # host mode: queued handles, oldest first
        self.stats = {"packed": 0, "kept": 0, "bytes_in": 0, "bytes_stored": 0}

    # ------------------------------------------------------------------ context manager
    def __enter__(self):
        torch = _torch()
        self._seen, self._order = {}, []  # a new forward pass
        self._hooks = torch.autograd.graph.saved_tensors_hooks(self._pack, self._unpack)
        self._hooks.__enter__()
        return self

    def __exit__(self, *exc):
        self._hooks.__exit__(*exc)
        self._hooks = None
        self._seen = {}
        return False

    # ------------------------------------------------------------------ buffers, streams
    def _workspace(self, device, nbytes, key=None):
        key = device if key is None else key
        with self._lock:
            ws = self._ws.get(key)
            if ws is None or ws.numel() < nbytes:
                if ws is not None:
                    self._keep.append(ws)
                ws = new_workspace(nbytes, device)
                self._ws[key] = ws
            return ws

    def _stream(self, table, device):
        with self._lock:
            s = table.get(device)
            if s is None:
                s = _torch().cuda.Stream(device=device)
                table[device] = s
            return s

    def _reap(self):
        """Drops retired pinned buffers whose last device use has completed."""
        with self._lock:
            self._retired = [(b, e) for b, e in self._retired if e is not None and not e.query()]

    # ------------------------------------------------------------------ hooks
    def _eligible(self, t):
        torch = _torch()
        return (isinstance(t, torch.Tensor) and t.is_cuda and t.element_size() == 4
                and t.numel() >= self.min_elems and t.is_contiguous()
                and not isinstance(t, torch.nn.Parameter))

    def _pack(self, t):
        if not self._eligible(t):
            self.stats["kept"] += 1
            return t
        # The same live tensor saved again reuses its handle. Memory freed during the
        # forward pass is handed to later tensors, so the address alone does not identify
        # a tensor: the entry also holds a weak reference to the tensor it was made for.
        key = (t.untyped_storage().data_ptr(), t.storage_offset(), tuple(t.shape), t._version)
        with self._lock:
            seen = self._seen.get(key)
            if seen is not None and seen[0]() is t:
                seen[1].saves += 1
                return seen[1]
            h = _Packed(t, len(self._order), self._order, weakref.ref(self))
            self._order.append(weakref.ref(h))
            self._seen[key] = (weakref.ref(t), h)
        torch = _torch()
        self._reap()
        stream = torch.cuda.current_stream(t.device)
        sh = stream.cuda_stream
        n, C = h.n, self.C
        if self.where == "host":
            cap = zvc_offload_host_bound(n, C)
            h.host = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
            produced = torch.cuda.Event()
            produced.record(stream)
            ws_stream = self._stream(self._wstream, t.device)
            t.record_stream(ws_stream)  # not reused before the worker's kernels have read it
            h.offloaded = threading.Event()
            while self._pending and self._pending[0].offloaded.is_set():
                self._pending.popleft()
            while len(self._pending) >= max(self.max_pending, 1):
                self._pending.popleft().offloaded.wait()
            self._submit((h, t, produced, cap))
            self._pending.append(h)
            if self.max_pending == 0:  # the loop waits for every tensor's offload
                h.offloaded.wait()
            self.stats["packed"] += 1
            self.stats["bytes_in"] += 4 * n
            return h
        else:
            cap = zvc_size_bound(n, C)
            ws = self._workspace(t.device, zvc_workspace_size(n, C))
            full = torch.empty(cap, dtype=torch.uint8, device=t.device)
            size = torch.zeros(1, dtype=torch.int64, device=t.device)
            _check(zvc_compress(t.data_ptr(), n, C, full.data_ptr(), cap, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), sh), "zvc_compress")
            h.size = int(size.item())  # waits for this tensor's compression
            h.dev = full[:h.size].clone()  # exactly the compressed bytes stay in HBM
        self.stats["packed"] += 1
        self.stats["bytes_in"] += 4 * n
        self.stats["bytes_stored"] += h.size
        return h

    def _submit(self, job):
        if self._worker is None:
            self._jobs = queue.Queue()
            self._worker = threading.Thread(target=_offload_worker,
                                            args=(weakref.ref(self), self._jobs), daemon=True)
            self._worker.start()
        self._jobs.put(job)

    def _offload_one(self, h, t, produced, cap):
        """On the worker thread: zvc_offload of one queued tensor (it blocks here, not in
        the training loop)."""
        torch = _torch()
        torch.cuda.set_device(h.device)
        ws_stream = self._stream(self._wstream, h.device)
        ws_stream.wait_event(produced)
        ws = self._workspace(h.device, zvc_offload_workspace_size(h.n, self.C),
                             key=("worker", h.device))
        st, size = zvc_offload(t.data_ptr(), h.n, self.C, h.host.data_ptr(), cap, ws.data_ptr(),
                               ws.numel(), ws_stream.cuda_stream)
        _check(st, "zvc_offload")
        # an event after this tensor's copies, without holding up any stream
        js = self._stream(self._join, h.device)
        _check(zvc_offload_join(js.cuda_stream), "zvc_offload_join")
        done = torch.cuda.Event()
        done.record(js)
        h.size, h.done = size, done
        with self._lock:
            self.stats["bytes_stored"] += size

    def close(self):
        """Stops the worker thread once the queued tensors are offloaded."""
        if self._worker is not None:
            self._jobs.put(None)
            self._worker.join()
            self._worker = self._jobs = None

    def __del__(self):
        jobs = getattr(self, "_jobs", None)  # absent if __init__ raised
        if jobs is not None:
            jobs.put(None)

    def _wait_offloaded(self, h):
        if h.offloaded is not None:
            h.offloaded.wait()
            if h.error is not None:
                raise h.error

    def _start_restore(self, h):
        """Enqueues the restore of h on the side stream; sets h.out and h.ready."""
        torch = _torch()
        side = self._stream(self._side, h.device)
        side.wait_stream(torch.cuda.current_stream(h.device))
        self._wait_offloaded(h)
        if h.done is not None:
            side.wait_event(h.done)  # the offload's copies have filled the host buffer
        with torch.cuda.stream(side):
            out = torch.empty(h.shape, dtype=h.dtype, device=h.device)
            sh = side.cuda_stream
            if self.where == "host":
                ws = self._workspace(h.device, zvc_offload_workspace_size(h.n, self.C))
                _check(zvc_prefetch(h.host.data_ptr(), h.size, out.data_ptr(), h.n, self.C,
                                    ws.data_ptr(), ws.numel(), sh), "zvc_prefetch")
            else:
                ws = self._workspace(h.device, 256)
                h.dev.record_stream(side)  # read here: not reused before this stream is done
                _check(zvc_decompress(h.dev.data_ptr(), h.size, out.data_ptr(), h.n, self.C,
                                      ws.data_ptr(), ws.numel(), sh), "zvc_decompress")
            h.ready = torch.cuda.Event()
            h.ready.record(side)
        h.out = out
        h.done = h.ready  # the restore's copies follow the offload's on the copy stream

    def _unpack(self, h):
        if not isinstance(h, _Packed):
            return h
        torch = _torch()
        main = torch.cuda.current_stream(h.device)
        if h.out is None:
            self._start_restore(h)
        main.wait_event(h.ready)
        out = h.out
        out.record_stream(main)
        h.unpacks += 1
        if h.unpacks % h.saves == 0:  # every operator that saved it has it: drop the copy
            h.out = None
        if self.prefetch_ahead and h.order > 0:
            prev = h.peers[h.order - 1]()
            if prev is not None and prev.out is None:
                self._start_restore(prev)
        return out

    def check_errors(self):
        """Raises if any kernel of this offloader latched a device-side error."""
        with self._lock:
            items = list(self._ws.items())
        for dev, ws in items:
            st = get_error(ws)
            if st != 0:
                raise ZvcError(st, f"device {dev}")
