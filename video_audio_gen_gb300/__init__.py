"""GB300-native packed-varlen joint video+audio DiT forward (libdit.so) and its Python binding.

Importing the package loads nothing; ``video_audio_gen_gb300.dit`` loads libdit.so on first use and
raises if it has not been built (``video_audio_gen_gb300.build.build()``).
"""
