"""Paged-KV decode step for GB300 (sm_103a): KV append, GQA paged decode attention
with split-KV, and the temperature / top-k / top-p / Philox sampler."""
