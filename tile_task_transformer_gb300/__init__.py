"""GB300-native tile-task GPT2 training step (forward, backward, fused AdamW).

The compute path is ``libnnt.so`` (CUDA for sm_103a behind a C ABI declared in
``include/nnt.h``); :mod:`tile_task_transformer_gb300.nnt` is its ctypes binding
and :mod:`tile_task_transformer_gb300.synth` holds the seeded input generators.
Importing the package itself loads nothing.
"""
