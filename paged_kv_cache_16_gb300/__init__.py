"""GB300-native data plane of one continuous-batching engine step.

The computation lives in ``libpa.so`` (hand-written CUDA for sm_103a behind
the C ABI of ``include/pa.h``); ``binding`` marshals arguments to it,
``step`` wires the calls of one step together for torch tensors, and
``workloads`` draws seeded synthetic batches.  Nothing here falls back to a
CPU or PyTorch implementation: without the compiled library the calls fail.
"""
from .binding import (PaError, Plan, load, pa_attention, pa_check_device_errors, pa_plan,  # noqa: F401
                      pa_plan_status, pa_slot_mapping, pa_write_kv, status_string)
