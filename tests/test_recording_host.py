"""ops.recording on the host: nesting is refused, a recording is per thread,
and recorded steps run in order (no GPU needed: only host callables)."""
import threading

import pytest

from paged_kv_cache_76_gb300 import ops


def test_steps_run_in_order_and_nesting_is_refused():
    seen = []
    with ops.recording() as rec:
        rec.add(lambda: seen.append(1))
        rec.add(lambda: seen.append(2))
        with pytest.raises(RuntimeError):
            with ops.recording():
                pass
    assert seen == []
    rec()
    rec()
    assert seen == [1, 2, 1, 2]


def test_a_recording_belongs_to_its_thread():
    state = {}
    with ops.recording() as rec:
        def other():
            state["other_open"] = getattr(ops._tls, "rec", None)
            with ops.recording() as r2:  # allowed: this thread has none open
                state["r2"] = r2
        th = threading.Thread(target=other)
        th.start()
        th.join()
        assert ops._tls.rec is rec
    assert state["other_open"] is None and state["r2"] is not rec
    assert getattr(ops._tls, "rec", None) is None
