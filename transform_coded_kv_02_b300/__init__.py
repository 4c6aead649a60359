"""Transform-coded KV cache for B300 (sm_103a).

    from transform_coded_kv_02_b300 import kvtc     # binding of the C-ABI library libkvtc.so
    from transform_coded_kv_02_b300 import synth    # seeded synthetic inputs (no codec arithmetic)
"""
