"""GB300-native mega-kernel decode runtime (tGraph builder + persistent
sm_103a kernel) behind the C-ABI library ``libmpk.so``.

``synth`` (seeded synthetic inputs) imports nothing else from this package;
the ctypes binding lives in ``task_graph_runtime_gb300.mpk`` and loads the
compiled library on first use, failing loudly when it is missing."""
