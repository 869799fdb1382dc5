"""The Python Hessian object may be shared by threads: its borrowed-batch
list is guarded by a lock, merges take the two objects' locks in one global
order, and no locked method calls another.  The C calls are replaced by
stand-ins here (no GPU), so only the binding's own locking is exercised."""

import threading

import torch

from gptq_qqq_calibration_gb300 import hessian as hz


def _fake_object(handle):
    h = hz.Hessian.__new__(hz.Hessian)
    h.d, h.handle, h._queued, h._lock = 8, handle, [], threading.Lock()
    return h


def test_shared_objects_do_not_deadlock(monkeypatch):
    pending = {}
    monkeypatch.setattr(hz, "hess_add_batch", lambda h, X, d, s=None: pending.__setitem__(h, pending.get(h, 0) + 1))
    monkeypatch.setattr(hz, "hess_pending_batches", lambda h: pending.get(h, 0))
    monkeypatch.setattr(hz, "hess_flush", lambda h, s=None: None)
    monkeypatch.setattr(hz, "hess_materialize", lambda h, out, damp, s=None, want=True: 0.0)
    monkeypatch.setattr(hz, "hess_reset", lambda h, s=None: pending.__setitem__(h, 0))
    monkeypatch.setattr(hz, "hess_merge", lambda a, b, s=None: None)
    monkeypatch.setattr(hz, "hess_clone", lambda h, s=None: 99)
    monkeypatch.setattr(hz, "hess_destroy", lambda h: None)
    a, b = _fake_object(1), _fake_object(2)
    out = torch.empty((8, 8))
    X = torch.ones((4, 8))

    def work(k):
        for i in range(200):
            h, o = (a, b) if (i + k) % 2 else (b, a)
            h.add_batch(X)
            h.flush()
            h.materialize(0.0, out=out, want_damp=False)
            h.merge(o)
            if i % 50 == 0:
                h.clone().close()
                h.reset()

    threads = [threading.Thread(target=work, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=60)
    assert not any(t.is_alive() for t in threads), "a lock was never released"
    assert len(a._queued) == pending.get(1, 0) and len(b._queued) == pending.get(2, 0)
