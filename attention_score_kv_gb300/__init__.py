"""Layer-end KV-cache compression by attention scoring on GB300 (sm_103a).

The CUDA library lives in ``libkvc.so`` (C ABI: ``include/kvc.h``); the
binding is :mod:`attention_score_kv_gb300.kvc`.  Build with
``python -m attention_score_kv_gb300.build``.
"""

__version__ = "0.1.0"
