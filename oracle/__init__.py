"""Plain CPU oracle for low-bit KV-cache append and decode attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg / reference arm of ``bench.py`` may import anything from
here. The product package never imports it and has no CPU fallback.

Two independent implementations of the same definitions:
  * ``oracle_cpp`` -- C++ (``kvq_oracle.cpp``), threaded over streams; the one
    used at full size and for the timed CPU baseline;
  * ``oracle_np``  -- NumPy, vectorized; used on small cases to cross-check the
    C++ one.
Every function is pinned by ``tests/test_oracle_pins.py`` to facts fixed by the
method and by mathematics (grid round trip, error bound, brute force,
closed forms, textbook softmax/rotation), not by re-calling itself.
"""
