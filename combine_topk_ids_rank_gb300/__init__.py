"""GB300-native top-k expert-parallel dispatch / combine on logical ranks.

The CUDA library is reached through `combine_topk_ids_rank_gb300.moe_a2a`
(a thin ctypes binding of the C ABI); importing the package itself loads
nothing.  `synth` draws the seeded synthetic inputs."""
